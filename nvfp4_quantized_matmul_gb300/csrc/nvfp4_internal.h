// Internal launchers shared between the C-ABI layer and the kernel files.
// Arguments are already validated by the caller (nvfp4_api.cu).
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

namespace nvfp4 {

enum XType : int { kF32 = 0, kF16 = 1, kBF16 = 2 };

cudaError_t launch_transcode(const uint8_t* mo_w, int64_t w_bytes, const uint8_t* mo_ws, int64_t s_bytes,
                             const float* ws2, uint32_t* w_out, uint8_t* s_out, float* gs_out,
                             cudaStream_t st);

cudaError_t launch_dequantize(const uint32_t* w, const uint8_t* scales, const float* gs, int64_t E,
                              int64_t N, int64_t K, int out_dtype, void* out, cudaStream_t st);
// Dense x [E, N, K] (f32, f16 or bf16) -> packed words and E4M3 block scales.
cudaError_t launch_quantize(const void* x, int x_dtype, const float* gs, int64_t E, int64_t N, int64_t K,
                            uint32_t* w, uint8_t* scales, cudaStream_t st);
// ModelOpt triplet -> packed words and folded E4M3 scales (no sidecar).
cudaError_t launch_transcode_folded(const uint8_t* mo_w, int64_t w_bytes, const uint8_t* mo_ws, int64_t s_bytes,
                                    const float* ws2, uint32_t* w_out, uint8_t* s_out, cudaStream_t st);
// Reads and clears the error code of the bulk-copy transcode's bounded waits.
int read_copy_error();

// Decode-shape product on the SIMT/mma.sync path. Row r of the output uses
// activation row lhs[r] (r when lhs is null) and expert rhs[r] (0 when rhs is
// null); rows whose expert is >= E or whose activation row is >= B are zero.
struct QmvArgs {
  const void* x;          // [B, K], dtype xdt
  const uint32_t* w;      // [E, N, K/8]
  const uint8_t* scales;  // [E, N, K/16]
  const float* gs;        // null or [E]
  const uint32_t* lhs;    // null or [R]
  const uint32_t* rhs;    // null or [R]
  int64_t B, R, K, N, E;
  void* y;                // [R, N], dtype xdt ([R, glu_cols] for a fused gate/up call)
  // Fused gate/up: w holds N = 2 * glu_cols rows (gate, then up) and y gets
  // act(gate) * up; glu_act 1 = SiLU, 2 = GELU (tanh form); 0 = plain call.
  int64_t glu_cols = 0;
  int glu_act = 0;
  // Batched weights: with rhs null, row r uses expert r / rows_per_expert
  // (the expert-group route only).
  int64_t rows_per_expert = 0;
};
cudaError_t launch_qmv(const QmvArgs& a, int xdt, cudaStream_t st);

// Largest K the 16-bit decode-shape route stages in shared memory (sixteen
// CTAs per cluster, eight rows per tile).
constexpr int64_t kQmvMaxK = 196608;
bool qmv_supported_k(int64_t K);
// TMA-fed variant of the decode-shape route (16-bit activations, K % 256 == 0).
bool qmv_tma_supported(const QmvArgs& a, int xdt);
cudaError_t launch_qmv_tma(const QmvArgs& a, int xdt, cudaStream_t st);
int read_qmv_error();
// Persistent stream-K decode route for dense QuantizedMatmul (16-bit
// activations, K % 256 == 0; one launch per 16 token rows). It finishes row tiles split
// between CTAs through a per-(device, stream) workspace that the library
// allocates on the first call on a stream (and grows on demand).
bool qmv_stream_supported(const QmvArgs& a, int xdt);
cudaError_t launch_qmv_stream(const QmvArgs& a, int xdt, cudaStream_t st);
int read_stream_error();
void release_stream_workspaces();
// The same kernel for GatherQMM with at most one row per SM (16-bit
// activations, K % 256 == 0): rows grouped by expert, eight to a group, each
// group's expert plane streamed once and split over its share of the SMs.
bool qmv_group_supported(const QmvArgs& a, int xdt);
// The dense route for a fused gate/up call (a.glu_act != 0): same limits as
// qmv_stream_supported.
cudaError_t launch_qmv_stream_glu(const QmvArgs& a, int xdt, cudaStream_t st);
cudaError_t launch_qmv_group(const QmvArgs& a, int xdt, cudaStream_t st);
// The same route with its scratch in a fixed array inside the library (no
// allocation); at most kNoAllocMaxRows weight rows.
constexpr int64_t kNoAllocMaxRows = 65536;
// cudaErrorInvalidConfiguration (nothing queued) when the decode kernel has
// no launch plan for the shape.
cudaError_t launch_qmv_stream_noalloc(const QmvArgs& a, int xdt, cudaStream_t st);
// Forgets the fixed array's device addresses (looked up again on next use).
void release_noalloc_addresses();

// A sequence of decode calls (16-bit x of dtype xdt, 1 <= M <= 16 rows each,
// K % 256 == 0) run by one persistent launch of the decode kernel, in order;
// call c with depends[c] != 0 (c > 0) reads its activations only after every
// earlier call has finished (cooperative launch). At most kSeqMaxCallsApi
// calls; the split-tile workspace is the stream's decode workspace.
constexpr int kSeqMaxCallsApi = 32;
bool qmv_seq_call_supported(const QmvArgs& a, int xdt);
cudaError_t launch_qmv_seq(const QmvArgs* calls, const int* depends, int n, int xdt, cudaStream_t st);

// Process-wide options set through nvfp4_set_option (include/nvfp4.h); each
// kernel family reads its own with option(). The values are those of the
// header's nvfp4_option enumeration.
enum Option : int {
  kOptTcTile = 1,
  kOptTcStreamK = 2,
  kOptNtDecode = 3,
  kOptQmvRowTiles = 4,
  kOptGatherGroup = 5,
  kOptGatherTc = 6,
  kOptGatherTile = 7,
  kOptWaitLimitUs = 8,
  kOptTestWithhold = 9,
  kOptEnd = 10
};
int option(int opt);

// Whether weight-streaming launches may overlap the previous kernel on the
// stream (programmatic dependent launch; see nvfp4_set_launch_overlap).
bool launch_overlap();

// Prefill-shape tensor-core route (tcgen05, TMEM accumulators).
bool qmm_tc_supported(int64_t M, int64_t N, int64_t K);
// Whether its dense launches split the last partial wave of tiles by k-blocks
// (stream-K; on unless the NVFP4_OPT_TC_STREAMK option is 0).
bool tc_stream_k();
cudaError_t launch_qmm_tc(const void* x, int xdt, int64_t M, int64_t K, const uint32_t* w, const uint8_t* scales,
                          const float* gs, int64_t N, void* y, cudaStream_t st);
// Fused gate/up on the tensor cores: w is [2 cols, K/8] (gate rows, then up
// rows), y [M, cols] = act(gate) * up; act 1 = SiLU, 2 = GELU (tanh form).
cudaError_t launch_qmm_tc_glu(const void* x, int xdt, int64_t M, int64_t K, const uint32_t* w, const uint8_t* scales,
                              const float* gs, int64_t cols, int act, void* y, cudaStream_t st);
// Non-transposed weights: w is [K, N/8] words quantized along N (N % 16 ==
// 0, any K >= 1), y = x @ dequantize(w) * gs/2688; f16 or bf16 x.
bool qmm_tc_nt_supported(int64_t M, int64_t N, int64_t K);
// Up to kQmvNtMaxM token rows of a non-transposed weight: one streaming pass
// over the plane per eight rows (the eight token rows are the eight columns
// of an m16n8k16 MMA's B operand, so any M up to 8 costs the same), partial
// sums in a per-stream float workspace, then y. Two passes (M = 9..16) still
// beat the tensor cores ([5376, 21504]: about 62 against 71 µs at M = 16).
constexpr int64_t kQmvNtMaxM = 16;
bool qmv_nt_supported(int64_t M, int64_t N, int64_t K);
cudaError_t launch_qmv_nt(const void* x, int xdt, int64_t M, int64_t K, const uint32_t* w, const uint8_t* scales,
                          const float* gs, int64_t N, void* y, cudaStream_t st);
void release_nt_workspaces();
cudaError_t launch_qmm_tc_nt(const void* x, int xdt, int64_t M, int64_t K, const uint32_t* w, const uint8_t* scales,
                             const float* gs, int64_t N, void* y, cudaStream_t st);
// Expert-batched GatherQMM on the tensor cores, for rows sorted by expert.
bool gather_tc_supported(int64_t B, int64_t K, int64_t R, int64_t E, int64_t N);
cudaError_t launch_gather_tc(const void* x, int xdt, int64_t B, int64_t K, const uint32_t* lhs, const uint32_t* rhs,
                             int64_t R, const uint32_t* w, const uint8_t* scales, const float* gs, int64_t E, int64_t N,
                             void* y, cudaStream_t st);
// Frees the gathered-activation buffers of the expert-batched route.
void release_gather_workspaces();
// Reads and clears the error code left by a bounded wait in the tensor-core
// kernels (synchronises with the device); 0 = none, -1 = read failed.
int read_tc_error();

}  // namespace nvfp4
