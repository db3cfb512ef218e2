/*
 * nvfp4.h - C ABI of libnvfp4.so, NVFP4 quantized matmul for NVIDIA GB300 (sm_103a).
 *
 * Weight format (mlxcel issue #693 "direct-transcode ModelOpt triplets to MLX
 * native", Technical notes):
 *   w       uint32 [E, N, K/8]  eight E2M1 codes per word along K; column
 *                               8*j+i of a row is nibble i of word j, counted
 *                               from the least significant nibble. E2M1 code
 *                               c has magnitude {0,.5,1,1.5,2,3,4,6}[c & 7]
 *                               and is negative when bit 3 is set.
 *   scales  uint8  [E, N, K/16] one E4M3 (OCP E4M3FN) byte per 16 columns.
 *   gs      float  [E] or none  optional global scale; outputs (and
 *                               dequantized elements) are multiplied by
 *                               gs[e] / (448 * 6) once (mlxcel PR #2629
 *                               "ROCm native NVFP4", Summary).
 * For a single linear E = 1. The scale plane must hold exactly
 * w.shape[:-1] + [w.shape[-1] / 2] bytes (PR #2629, Changes during review);
 * lengths are passed so the library can refuse a mismatched plane.
 *
 * Conventions for every entry point:
 *   - All data pointers are DEVICE pointers owned by the caller; the library
 *     keeps no reference after the call returns. Lengths are element counts.
 *   - Work is enqueued asynchronously on `stream` (a cudaStream_t; NULL is the
 *     legacy default stream). Nothing is synchronised. The library allocates
 *     three kinds of scratch, each one per (device, stream): the decode
 *     route's split-tile workspace (see nvfp4_qmm), the tensor-core route's
 *     stream-K sums (up to two waves of 256 x 256 f32 tiles and a counter
 *     each, about 78 MB on 152 SMs) and the expert-batched gather's row
 *     buffer (see nvfp4_gather_qmm). Each is made on the first call on a
 *     stream that needs it, or the first that needs more, and kept until
 *     nvfp4_shutdown(). Made while the stream is being captured into a CUDA
 *     graph, the allocation is done outside the capture (the thread's capture
 *     mode relaxed for it) and the graph uses that memory on every replay.
 *   - Data pointers must be 16-byte aligned; index arrays and gs 4-byte.
 *   - K must be a multiple of 16. Any N >= 1 is accepted.
 *   - Empty outputs (M, N or R equal to 0) return NVFP4_OK without a launch.
 *   - On failure nothing is launched (validation errors) or the CUDA launch
 *     error is returned as NVFP4_ERR_CUDA; nvfp4_last_error() then holds a
 *     message for the calling thread.
 */
#ifndef NVFP4_H
#define NVFP4_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  NVFP4_OK = 0,
  NVFP4_ERR_NULL = 1,    /* a required pointer is NULL */
  NVFP4_ERR_SHAPE = 2,   /* negative size, K % 16 != 0, size overflow */
  NVFP4_ERR_PLANE = 3,   /* weight or scale plane length does not match the shape */
  NVFP4_ERR_DTYPE = 4,   /* unknown dtype or route */
  NVFP4_ERR_ALIGN = 5,   /* pointer not aligned as required */
  NVFP4_ERR_GSCALE = 6,  /* gs given with the wrong length (or a length without gs) */
  NVFP4_ERR_LIMIT = 7,   /* launch dimensions beyond what the kernels support */
  NVFP4_ERR_CUDA = 8     /* CUDA reported an error at launch */
} nvfp4_status;

typedef enum { NVFP4_F32 = 0, NVFP4_F16 = 1, NVFP4_BF16 = 2 } nvfp4_dtype;

/* Route for nvfp4_qmm_routed: AUTO picks by the measured M crossover. */
typedef enum { NVFP4_ROUTE_AUTO = 0, NVFP4_ROUTE_QMV = 1, NVFP4_ROUTE_TC = 2 } nvfp4_route;

/*
 * ModelOpt triplet -> native planes (issue #693, Goal and Implementation plan
 * step 3): four source bytes become one little-endian uint32, the E4M3 block
 * scales are kept byte for byte, and weight_scale_2 becomes the global-scale
 * sidecar gs = ws2 * 2688 (float32 multiply), so that the native factor
 * gs / 2688 stands for ws2. No dense intermediate is formed.
 *   mo_weight        uint8 [N, K/2]   two E2M1 codes per byte, low nibble = even column
 *   mo_weight_scale  uint8 [N, K/16]  E4M3
 *   weight_scale_2   float [1]        device scalar
 *   w_out [N, K/8] uint32, scales_out [N, K/16] uint8, gs_out float [1]
 * Lengths must equal N*K/2 and N*K/16 (NVFP4_ERR_PLANE otherwise). The
 * planes are moved by bulk copies through shared memory (one CTA per SM).
 */
nvfp4_status nvfp4_transcode(const uint8_t* mo_weight, int64_t mo_weight_len, const uint8_t* mo_weight_scale,
                             int64_t mo_weight_scale_len, const float* weight_scale_2, int64_t N, int64_t K,
                             uint32_t* w_out, uint8_t* scales_out, float* gs_out, void* stream);

/*
 * Folded-scale transcode, the alternative issue #693 (Technical notes)
 * rejects: weight_scale * weight_scale_2 folded into every E4M3 block scale
 * and no sidecar, built to measure the overflow and rounding drift that the
 * sidecar avoids (dequantize the result with gs NULL and compare it with the
 * sidecar transcode). Weight bytes as nvfp4_transcode; each scale byte
 * becomes the E4M3 value nearest to f32(e4m3(b) * ws2), ties to even,
 * saturating at 448, products below 2^-10 flushed to 0. Non-negative finite
 * scale bytes only (others give unspecified bytes, no fault).
 *   mo_weight uint8 [N, K/2], mo_weight_scale uint8 [N, K/16],
 *   weight_scale_2 float [1] on the device; w_out [N, K/8], scales_out
 *   [N, K/16]. Lengths and refusals as nvfp4_transcode.
 */
nvfp4_status nvfp4_transcode_folded(const uint8_t* mo_weight, int64_t mo_weight_len, const uint8_t* mo_weight_scale,
                                    int64_t mo_weight_scale_len, const float* weight_scale_2, int64_t N, int64_t K,
                                    uint32_t* w_out, uint8_t* scales_out, void* stream);

/*
 * Exact dequantize (PR #2629, Summary; Changes during review: sized from the
 * weight plane). out[e, n, k] = cast_rne(f32(fp4 * e4m3) * f32(gs[e] / 2688)),
 * or the exact product when gs is NULL. out is [E, N, K] of out_dtype.
 * gs_len must be 0 (gs NULL) or E.
 */
nvfp4_status nvfp4_dequantize(const uint32_t* w, int64_t w_len, const uint8_t* scales, int64_t scales_len,
                              const float* gs, int64_t gs_len, int64_t E, int64_t N, int64_t K,
                              nvfp4_dtype out_dtype, void* out, void* stream);

/*
 * Dense -> NVFP4 quantize, the encoding half of MLX's global-scale convention
 * (PR #2629, Implementation Review Summary: fp_quantize encodes block scales
 * times 448 * 6 / global_scale; issue #693, Context: the dense f16 -> MLX
 * quantize(mode="nvfp4") repair path). For each run of 16 columns, in IEEE
 * float32 with round to nearest even:
 *   amax = max |x|;  s = amax / 6, times 2688 / gs[e] when gs is given;
 *   scale byte = the E4M3 value nearest to s, ties to even, saturating at 448;
 *   d = e4m3(scale byte) * gs[e] / 2688 (the multiplier dequantize applies);
 *   code = the E2M1 value nearest to x * (1 / d), ties to even, saturating at
 *          +-6, +0 where the magnitude rounds to 0, every code 0 where d == 0.
 * The rounding and saturation rules are this library's reading; the pages
 * do not state them. NaN or infinite inputs give unspecified codes (no
 * fault). With gs[e] = max |x[e]| every block scale is at most 448 and
 * nothing saturates; without gs a block whose amax exceeds 2688 saturates.
 *   x [E, N, K] of x_dtype (16-byte aligned), gs NULL (gs_len 0) or E floats
 *   on the device (positive and finite), w [E, N, K/8] uint32 and scales
 *   [E, N, K/16] uint8 written (lengths as for nvfp4_dequantize;
 *   NVFP4_ERR_PLANE otherwise). K % 16 == 0.
 */
nvfp4_status nvfp4_quantize(const void* x, nvfp4_dtype x_dtype, int64_t E, int64_t N, int64_t K, const float* gs,
                            int64_t gs_len, uint32_t* w, int64_t w_len, uint8_t* scales, int64_t scales_len,
                            void* stream);

/*
 * QuantizedMatmul (PR #2629, Summary): y = x @ dequantize(w).T, with the
 * global factor gs / 2688 applied once per output after the f32 sum.
 *   x [M, K] of x_dtype (f32, f16 or bf16), w [N, K/8], scales [N, K/16],
 *   gs NULL (gs_len 0) or one float (gs_len 1), y [M, N] of x_dtype.
 * The route (decode-shape qmv or the tcgen05 tensor-core path) is chosen by
 * comparing M with nvfp4_qmm_crossover().
 * With 16-bit activations, 1 <= M <= 16 and K % 256 == 0 the decode route
 * splits the weight plane evenly over the SMs; a 256-row block of outputs
 * computed by several CTAs is summed in a float32 workspace owned by the
 * library, one per (device, stream): 64 bytes per weight row plus a counter
 * per 256 rows, returned to zero by every call that completes. Calls on one
 * stream are ordered, so they never share it concurrently.
 */
nvfp4_status nvfp4_qmm(const void* x, nvfp4_dtype x_dtype, int64_t M, int64_t K, const uint32_t* w,
                       int64_t w_len, const uint8_t* scales, int64_t scales_len, const float* gs,
                       int64_t gs_len, int64_t N, void* y, void* stream);

/* nvfp4_qmm with an explicit route (tests and crossover sweeps). */
nvfp4_status nvfp4_qmm_routed(const void* x, nvfp4_dtype x_dtype, int64_t M, int64_t K, const uint32_t* w,
                              int64_t w_len, const uint8_t* scales, int64_t scales_len, const float* gs,
                              int64_t gs_len, int64_t N, void* y, nvfp4_route route, void* stream);

/*
 * QuantizedMatmul with a non-transposed weight (PR #2629, Changes during
 * review and Review findings: the quantized axis of such a weight is N, so
 * the multiple-of-16 rule moves from K to N and x [1, 17] against a [17, 32]
 * weight is valid): y = x @ dequantize(w) * gs / 2688.
 *   x [M, K] of x_dtype (f16 or bf16; f32 is refused with ERR_DTYPE), any
 *   K >= 0; w [K, N/8] uint32 words, word j of row k holding outputs
 *   8j..8j+7 of input k (low nibble first); scales [K, N/16] E4M3 bytes, one
 *   per 16 outputs of an input; gs NULL (gs_len 0) or one float; y [M, N] of
 *   x_dtype. N % 16 == 0 (ERR_SHAPE otherwise). x, y, w and scales 16-byte
 *   aligned (ERR_ALIGN). M == 0 or N == 0 returns OK without a launch; K == 0
 *   writes zeros.
 * Up to sixteen token rows: one streaming pass over the plane per eight rows
 * (m16n8k16 MMAs on nibble-interleaved pairs of input rows; each warp a run
 * of 16-input steps of one 256-output slab), partial sums added into a float
 * workspace [16, N] owned by the library, one per (device, stream), returned to zero by
 * every call; then y. More rows (or the NVFP4_OPT_NT_DECODE option set to
 * 0): the tcgen05 tensor-core
 * kernel, whose producer warps decode and transpose the weight tiles into
 * shared memory (the pages send every M to dequantize + GEMM). With
 * K % 8 != 0 the tensor-core route first copies the activations, rows padded
 * with zeros to a multiple of 8 elements, into the per-stream buffer of the
 * gathered activations (grown on demand, freed by nvfp4_shutdown()).
 */
nvfp4_status nvfp4_qmm_nontransposed(const void* x, nvfp4_dtype x_dtype, int64_t M, int64_t K, const uint32_t* w,
                                     int64_t w_len, const uint8_t* scales, int64_t scales_len, const float* gs,
                                     int64_t gs_len, int64_t N, void* y, void* stream);

/*
 * QuantizedMatmul with batched weights (PR #2629 "ROCm native NVFP4",
 * Numerical results: "qmm batched w"): y[b] = x[b] @ dequantize(w[b]).T *
 * gs[b] / 2688 for b < batches.
 *   x [batches, M, K] of x_dtype; w [batches, N, K/8]; scales [batches, N,
 *   K/16]; gs NULL (gs_len 0) or [batches]; y [batches, M, N] of x_dtype.
 * Below the crossover (16-bit x, K % 256 == 0, batches * M at most one row
 * per SM) all batches go out as one launch of the expert-group decode route;
 * otherwise one nvfp4_qmm per batch. Same refusals as nvfp4_qmm, with the
 * plane lengths and gs_len checked per batch count.
 */
nvfp4_status nvfp4_qmm_batched(const void* x, nvfp4_dtype x_dtype, int64_t batches, int64_t M, int64_t K,
                               const uint32_t* w, int64_t w_len, const uint8_t* scales, int64_t scales_len,
                               const float* gs, int64_t gs_len, int64_t N, void* y, void* stream);

/* Activation of the fused gate/up projection (nvfp4_qmm_glu). */
typedef enum { NVFP4_ACT_SILU = 1, NVFP4_ACT_GELU_TANH = 2 } nvfp4_act;

/*
 * Fused gate/up projection with its activation (issue #705 "close native
 * NVFP4 prefill gap", Hypothesis and Activation-path follow-up: the gated
 * MLP's GeGLU activation applied to the fused, globally scaled gate/up
 * projection, here fused into the matmul's epilogue):
 *   [g | u] = x @ dequantize(w).T * gs / 2688,   y = act(g) * u
 *   x [M, K] f16 or bf16; w [2 I, K/8] with the I gate rows first and the I
 *   up rows after them; scales [2 I, K/16]; gs NULL or one float; y [M, I]
 *   of x's dtype. act: SiLU (v * sigmoid(v)) or GELU in its tanh form
 *   (Gemma's GeGLU), evaluated in f32 on the f32 sums.
 * The intermediate [M, 2 I] never exists in memory. Below the crossover of
 * the [2 I, K] plane (or with route NVFP4_ROUTE_QMV) the decode route runs
 * (K % 256 == 0 required); otherwise the tensor-core route (K % 32 == 0),
 * whole tiles only. f32 activations are refused (NVFP4_ERR_DTYPE). Not an
 * interface of the pages; their follow-up names this fusion as the missing
 * prefill piece.
 */
nvfp4_status nvfp4_qmm_glu(const void* x, nvfp4_dtype x_dtype, int64_t M, int64_t K, const uint32_t* w,
                           int64_t w_len, const uint8_t* scales, int64_t scales_len, const float* gs,
                           int64_t gs_len, int64_t I, nvfp4_act act, void* y, nvfp4_route route, void* stream);

/*
 * nvfp4_qmm for callers that must not allocate device memory: a runtime whose
 * memory is planned once at start-up, or code that runs while a CUDA graph is
 * captured in the strict mode, where an allocation would break the capture.
 * Same arguments and result as nvfp4_qmm, always on the decode route; its
 * scratch is a fixed array inside the library (4 MB plus 1 KB, held on every
 * GPU that loads the library until the process exits). Limits: f16 or bf16
 * activations, 1 <= M <= 16, K a multiple of 256 (at most 2^20), N at most
 * 65536; other shapes, and shapes for which the decode kernel has no launch
 * plan, are refused (NVFP4_ERR_DTYPE / _SHAPE / _LIMIT) before anything is
 * queued. Nothing is allocated: the first call on a device looks up the
 * array's device address (make that call before any stream capture), and
 * every call clears the part of the array it uses on `stream` before its
 * kernel (the tile counters and, per 256-row tile, the M token slots of
 * sums: two memset nodes). All calls share the one array, so calls whose
 * work overlaps on the GPU (on different streams) race and give wrong
 * results: order them. nvfp4_shutdown() forgets the looked-up addresses;
 * call it before resetting a device's context, since an address from the
 * old context would be stale. The pages have no counterpart of this entry
 * point.
 */
nvfp4_status nvfp4_qmm_noalloc(const void* x, nvfp4_dtype x_dtype, int64_t M, int64_t K, const uint32_t* w,
                               int64_t w_len, const uint8_t* scales, int64_t scales_len, const float* gs,
                               int64_t gs_len, int64_t N, void* y, void* stream);

/* One QuantizedMatmul of a sequence (nvfp4_qmm_sequence): the arguments of
 * nvfp4_qmm for one call, y [M, N] = x [M, K] @ dequantize(w).T * gs / 2688. */
typedef struct {
  const void* x;          /* [M, K], the sequence's activation dtype */
  int64_t M, K, N;
  const uint32_t* w;      /* [N, K/8] packed E2M1 words */
  int64_t w_len;          /* words in w */
  const uint8_t* scales;  /* [N, K/16] E4M3 block scales */
  int64_t scales_len;     /* bytes in scales */
  const float* gs;        /* NULL (gs_len 0) or one float (gs_len 1) */
  int64_t gs_len;
  void* y;                /* [M, N], the activation dtype */
  /* Nonzero: this call reads x only once every earlier call of the sequence
   * has finished (set it when x is, or depends on, an earlier call's y). */
  int32_t after_previous;
  int32_t reserved;       /* set to 0 */
} nvfp4_qmm_call;

/*
 * A sequence of decode-shape QuantizedMatmuls (PR #2629, Summary: qmv for
 * small M, the global scale applied once per output) run in order by one
 * persistent launch on `stream`; the result is that of calling nvfp4_qmm on
 * each in turn. The calls of a decode step (the projections of a layer, at
 * one or several token counts) then share one weight-streaming pipeline:
 * the next call's weights stream while the current call's last tiles finish,
 * so the start and end of a launch are paid once per sequence instead of
 * once per call. Every call: f16 or bf16 activations (x_dtype, all calls),
 * 1 <= M <= 16 (M = 0 or N = 0 calls are skipped), K a positive multiple of
 * 256 (at most 2^20), N < 2^31; at most 32 calls. Other shapes are refused
 * (NVFP4_ERR_DTYPE / _SHAPE / _LIMIT / _PLANE / _GSCALE / _NULL / _ALIGN, the
 * message naming the call) before anything is queued.
 * Calls without after_previous must not read what earlier calls of the
 * sequence write (their activations are read while those calls may still
 * run). A call with after_previous waits, on the device, until every CTA has
 * finished every earlier call; the launch is then cooperative (all CTAs
 * resident at once) and each such wait gives up after 2 s with the error
 * code that nvfp4_take_device_error() reports. The weight planes of all
 * calls are read while earlier calls run: no call may write them. Scratch is
 * the stream's decode workspace (see nvfp4_qmm), grown on the first call
 * that needs more. Not an interface of the pages: it is this library's way
 * to run the several small-M matmuls of a decode step.
 */
nvfp4_status nvfp4_qmm_sequence(const nvfp4_qmm_call* calls, int32_t ncalls, nvfp4_dtype x_dtype, void* stream);

/* Smallest M routed to the tensor-core path for this shape and dtype. The
 * environment variable NVFP4_QMM_CROSSOVER overrides it. */
int64_t nvfp4_qmm_crossover(nvfp4_dtype x_dtype, int64_t N, int64_t K);

/*
 * GatherQMM (PR #2629, Summary; Changes during review):
 *   y[r] = x[lhs[r]] @ dequantize(w[rhs[r]]).T * gs[rhs[r]] / 2688
 *   x [B, K] of x_dtype; lhs_indices uint32 [R] or NULL (row r uses x[r]);
 *   rhs_indices uint32 [R]; w [E, N, K/8]; scales [E, N, K/16];
 *   gs NULL (gs_len 0) or [E] (gs_len E); y [R, N] of x_dtype.
 * A row whose expert index is >= E, or whose activation index is >= B, is
 * written as exact +0.0 (no read outside x or w). Calls with 16-bit
 * activations, K % 256 == 0 and at most one row per SM group the rows by
 * expert (eight to a group, in row order) and stream each group's expert
 * plane once, split over the SMs; they use the decode route's workspace (see
 * nvfp4_qmm). The NVFP4_OPT_GATHER_GROUP option set to 0 sends them to the
 * per-row kernel instead.
 * `sorted_indices` != 0
 * promises expert indices in non-decreasing order (a sorted MoE prefill) and
 * lets 16-bit calls with enough rows per expert (R >= 512 and R >= 16 E, E <=
 * 1024, K % 32 == 0) take the expert-batched tensor-core route; the
 * NVFP4_OPT_GATHER_TC option forces (1) or disables (0) that route.
 * With lhs_indices that route first copies the activation rows into output
 * order, in a buffer of R * K * 2 bytes that the library keeps per (device,
 * stream) until nvfp4_shutdown() (made outside any capture, as the decode
 * workspace).
 * If the promise is broken on that route, every output row is still written
 * once and nothing outside the inputs is read, but rows are computed with
 * the expert of the sorted segment they fall in.
 */
nvfp4_status nvfp4_gather_qmm(const void* x, nvfp4_dtype x_dtype, int64_t B, int64_t K, const uint32_t* lhs_indices,
                              const uint32_t* rhs_indices, int64_t R, int sorted_indices, const uint32_t* w,
                              int64_t w_len, const uint8_t* scales, int64_t scales_len, const float* gs,
                              int64_t gs_len, int64_t E, int64_t N, void* y, void* stream);

/* Error code recorded on the device by a pipelined kernel whose bounded
 * wait on a pipeline barrier ran out (each wait gives up after 2 s instead of
 * hanging, and the kernel then returns without finishing its tiles); the
 * call reads and clears it (and, after an error, clears the decode
 * workspaces). Blocks until all prior work on the current device
 * has finished. Returns 0 when no wait gave up, -1 if the read failed. Not
 * part of the pages' interface: it exists so that a kernel can report a stall
 * instead of holding the GPU. */
int32_t nvfp4_take_device_error(void);

/* Launch overlap for the weight-streaming calls (nvfp4_qmm below the
 * tensor-core crossover, nvfp4_gather_qmm). When enabled (non-zero) they are
 * launched as programmatic dependents of the kernel before them on the
 * stream: their CTAs may start, and begin streaming the weight and scale
 * planes, while that kernel is still finishing. Activations, indices and
 * outputs are touched only after it has completed and its writes are visible.
 * The caller promises that no kernel still running on the stream writes the
 * weight or scale planes (for example a transcode of those planes issued just
 * before). Off by default; process-wide. Returns the previous setting. Not
 * part of the pages' interface: it removes the idle gap between consecutive
 * decode-step matmuls, whose weights are constant. */
int nvfp4_set_launch_overlap(int enable);

/* Process-wide choices between equivalent kernels, for tests and tuning; the
 * defaults are the automatic choices and results agree to the stated
 * tolerances whatever is set. Not part of the pages' interface. */
typedef enum {
  NVFP4_OPT_TC_TILE = 1,        /* prefill tile: 0 automatic (default), 1 256x256, 2 256x128, 3 128x256 */
  NVFP4_OPT_TC_STREAMK = 2,     /* 1 (default): fewer than two waves of prefill tiles, the second at most 60%
                                   full, are split by k-blocks over all SMs; 0: whole tiles only */
  NVFP4_OPT_NT_DECODE = 3,      /* 1 (default): up to sixteen rows of a non-transposed weight take the streaming
                                   kernel; 0: the tensor cores */
  NVFP4_OPT_QMV_ROW_TILES = 4,  /* 16-row weight tiles per decode consumer warp: 0 automatic (default), 1, 2 */
  NVFP4_OPT_GATHER_GROUP = 5,   /* 1 (default): decode-shape gathers grouped by expert; 0: the per-row kernel */
  NVFP4_OPT_GATHER_TC = 6,      /* -1 automatic (default); 1: sorted gathers take the expert-batched
                                   tensor-core route wherever supported; 0: never */
  NVFP4_OPT_GATHER_TILE = 7,    /* expert-batched route's tile: 0 automatic (default, 256x256), 1 256x256,
                                   2 256x128, 3 128x256 */
  NVFP4_OPT_WAIT_LIMIT_US = 8,  /* decode-route calls of nvfp4_qmm: limit of each bounded wait in
                                   microseconds, 0 (default) for 2 s; for tests of the stall path */
  NVFP4_OPT_TEST_WITHHOLD = 9   /* tests of the stall path only: 1 makes the first CTA of the next
                                   decode-route nvfp4_qmm launches withhold the release of one
                                   pipeline stage, so that a bounded wait runs out (the call then
                                   reports its error code through nvfp4_take_device_error and
                                   leaves no copy in flight); 0 (default) off */
} nvfp4_option;

/* Sets an option: NVFP4_ERR_DTYPE for an unknown option, NVFP4_ERR_LIMIT
 * for a value outside its range (nothing changed). Takes effect for calls
 * made afterwards (a CUDA graph keeps the kernels it captured). */
nvfp4_status nvfp4_set_option(nvfp4_option option, int32_t value);
/* The option's current value (INT32_MIN for an unknown option). */
int32_t nvfp4_get_option(nvfp4_option option);

/* Frees the library's scratch (decode workspaces, stream-K sums, gathered-row
 * buffers) on every device. Call only when no
 * library work is queued or running; a later call allocates again. Not part
 * of the pages' interface. */
void nvfp4_shutdown(void);

/* Message for the calling thread's last non-OK status ("" if none). */
const char* nvfp4_last_error(void);

/* Library version string. */
const char* nvfp4_version(void);

#ifdef __cplusplus
}
#endif

#endif /* NVFP4_H */
