// C-ABI layer of libnvfp4.so: argument validation, route selection, launch.
//
// Validation follows the refusals on the pages (mlxcel PR #2629 "ROCm native
// NVFP4", Summary and Changes during review): a scale plane must hold exactly
// w.shape[:-1] + [w.shape[-1] / 2] bytes, K must be a multiple of 16, a
// global scale must have one entry per expert, an unexpected global-scale
// input is refused rather than ignored, launch limits are refused with a
// clear error, and empty outputs return before any launch.
#include <atomic>
#include <cinttypes>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <string>

#include "../../include/nvfp4.h"
#include "nvfp4_internal.h"

namespace {

thread_local std::string g_last_error;

nvfp4_status fail(nvfp4_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return s;
}

nvfp4_status ok() {
  g_last_error.clear();
  return NVFP4_OK;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// a * b without signed overflow, for non-negative operands.
bool mul_ok(int64_t a, int64_t b, int64_t* out) {
  if (a < 0 || b < 0) return false;
  if (a != 0 && b > INT64_MAX / a) return false;
  *out = a * b;
  return true;
}

int dtype_size(nvfp4_dtype d) { return d == NVFP4_F32 ? 4 : 2; }
bool dtype_ok(nvfp4_dtype d) { return d == NVFP4_F32 || d == NVFP4_F16 || d == NVFP4_BF16; }

// Shared checks for a weight plane [E, N, K/8] with scales [E, N, K/16].
nvfp4_status check_planes(const char* fn, const uint32_t* w, int64_t w_len, const uint8_t* scales,
                          int64_t scales_len, int64_t E, int64_t N, int64_t K) {
  if (E < 0 || N < 0 || K < 0) return fail(NVFP4_ERR_SHAPE, "%s: negative size (E=%" PRId64 ", N=%" PRId64 ", K=%" PRId64 ")", fn, E, N, K);
  if (K % 16) return fail(NVFP4_ERR_SHAPE, "%s: K=%" PRId64 " is not a multiple of 16", fn, K);
  int64_t en, words, groups, elems;
  if (!mul_ok(E, N, &en) || !mul_ok(en, K, &elems) || !mul_ok(elems, 4, &elems))
    return fail(NVFP4_ERR_SHAPE, "%s: E*N*K overflows", fn);
  words = en * (K / 8);
  groups = en * (K / 16);
  if (w_len != words)
    return fail(NVFP4_ERR_PLANE, "%s: weight plane has %" PRId64 " words, expected E*N*K/8 = %" PRId64, fn, w_len, words);
  if (scales_len != groups)
    return fail(NVFP4_ERR_PLANE,
                "%s: scale plane has %" PRId64 " bytes, expected E*N*K/16 = %" PRId64
                " (scales.shape must be w.shape[:-1] + [w.shape[-1]/2])",
                fn, scales_len, groups);
  if (words > 0 && (!w || !scales)) return fail(NVFP4_ERR_NULL, "%s: weight or scale plane is NULL", fn);
  if (!aligned(w, 16) || !aligned(scales, 16)) return fail(NVFP4_ERR_ALIGN, "%s: weight/scale planes must be 16-byte aligned", fn);
  return NVFP4_OK;
}

nvfp4_status check_gs(const char* fn, const float* gs, int64_t gs_len, int64_t expect) {
  if (!gs) {
    if (gs_len != 0) return fail(NVFP4_ERR_GSCALE, "%s: gs is NULL but gs_len=%" PRId64, fn, gs_len);
    return NVFP4_OK;
  }
  if (gs_len != expect)
    return fail(NVFP4_ERR_GSCALE, "%s: gs has %" PRId64 " entries, expected %" PRId64, fn, gs_len, expect);
  if (!aligned(gs, 4)) return fail(NVFP4_ERR_ALIGN, "%s: gs must be 4-byte aligned", fn);
  return NVFP4_OK;
}

nvfp4_status cuda_status(const char* fn, cudaError_t e) {
  if (e != cudaSuccess) return fail(NVFP4_ERR_CUDA, "%s: CUDA error %s (%s)", fn, cudaGetErrorName(e), cudaGetErrorString(e));
  return ok();
}

constexpr int64_t kMaxGridX = 0x7FFFFFFF;
constexpr int64_t kMaxGridY = 65535;

nvfp4_status check_qmv_grid(const char* fn, int64_t R, int64_t N) {
  if ((N + 15) / 16 > kMaxGridX || (R + 7) / 8 > kMaxGridY * 64)
    return fail(NVFP4_ERR_LIMIT, "%s: R=%" PRId64 ", N=%" PRId64 " exceed the launch limits", fn, R, N);
  return NVFP4_OK;
}

// Launch the decode-shape kernel in row blocks so grid.y stays within 65535.
cudaError_t run_qmv(nvfp4::QmvArgs a, int xdt, cudaStream_t st) {
  const int64_t chunk = kMaxGridY * 8;  // rows per launch: a multiple of every row tile
  const int64_t R = a.R;
  if (R <= chunk) return nvfp4::launch_qmv(a, xdt, st);
  const int64_t xsz = xdt == NVFP4_F32 ? 4 : 2;
  for (int64_t r = 0; r < R; r += chunk) {
    nvfp4::QmvArgs b = a;
    b.R = R - r < chunk ? R - r : chunk;
    b.y = static_cast<char*>(a.y) + r * a.N * xsz;
    if (a.lhs) b.lhs = a.lhs + r;
    if (a.rhs) b.rhs = a.rhs + r;
    if (!a.lhs) {  // identity activation rows: shift x instead
      b.x = static_cast<const char*>(a.x) + r * a.K * xsz;
      b.B = a.B - r;
    }
    cudaError_t e = nvfp4::launch_qmv(b, xdt, st);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

// Smallest M sent to the tensor-core route by default (measured sweep).
constexpr int64_t kDefaultCrossover = 128;

int64_t env_crossover() {
  const char* s = std::getenv("NVFP4_QMM_CROSSOVER");
  if (!s || !*s) return -1;
  char* end = nullptr;
  const long long v = std::strtoll(s, &end, 10);
  return (end && *end == 0 && v >= 0) ? (int64_t)v : -1;
}

}  // namespace

namespace nvfp4 {
std::atomic<int> g_launch_overlap{0};
bool launch_overlap() { return g_launch_overlap.load(std::memory_order_relaxed) != 0; }

namespace {
// Index: nvfp4_option value (0 unused). Defaults: automatic choices.
std::atomic<int> g_options[kOptEnd] = {0, 0, 1, 1, 0, 1, -1, 0, 0, 0};
constexpr int kOptMin[kOptEnd] = {0, 0, 0, 0, 0, 0, -1, 0, 0, 0};
constexpr int kOptMax[kOptEnd] = {0, 3, 1, 1, 2, 1, 1, 3, 2000000, 1};
}  // namespace

int option(int opt) { return g_options[opt].load(std::memory_order_relaxed); }
}  // namespace nvfp4

extern "C" {

const char* nvfp4_last_error(void) { return g_last_error.c_str(); }

const char* nvfp4_version(void) { return "nvfp4-gb300 0.1 (sm_103a)"; }

int nvfp4_set_launch_overlap(int enable) { return nvfp4::g_launch_overlap.exchange(enable ? 1 : 0); }

int32_t nvfp4_take_device_error(void) {
  const int a = nvfp4::read_tc_error(), b = nvfp4::read_qmv_error(), c = nvfp4::read_stream_error(),
            d = nvfp4::read_copy_error();
  if (a < 0 || b < 0 || c < 0 || d < 0) return -1;
  return a ? a : b ? b : c ? c : d;
}

nvfp4_status nvfp4_set_option(nvfp4_option option, int32_t value) {
  const int o = (int)option;
  if (o <= 0 || o >= nvfp4::kOptEnd)
    return fail(NVFP4_ERR_DTYPE, "nvfp4_set_option: unknown option %d", o);
  if (value < nvfp4::kOptMin[o] || value > nvfp4::kOptMax[o])
    return fail(NVFP4_ERR_LIMIT, "nvfp4_set_option: value %d of option %d outside %d..%d", (int)value, o,
                nvfp4::kOptMin[o], nvfp4::kOptMax[o]);
  nvfp4::g_options[o].store((int)value, std::memory_order_relaxed);
  return ok();
}

int32_t nvfp4_get_option(nvfp4_option option) {
  const int o = (int)option;
  if (o <= 0 || o >= nvfp4::kOptEnd) return INT32_MIN;
  return nvfp4::option(o);
}

void nvfp4_shutdown(void) {
  nvfp4::release_stream_workspaces();
  nvfp4::release_gather_workspaces();
  nvfp4::release_nt_workspaces();
  nvfp4::release_noalloc_addresses();
}

nvfp4_status nvfp4_transcode(const uint8_t* mo_weight, int64_t mo_weight_len, const uint8_t* mo_weight_scale,
                             int64_t mo_weight_scale_len, const float* weight_scale_2, int64_t N, int64_t K,
                             uint32_t* w_out, uint8_t* scales_out, float* gs_out, void* stream) {
  const char* fn = "nvfp4_transcode";
  if (N < 0 || K < 0) return fail(NVFP4_ERR_SHAPE, "%s: negative size", fn);
  if (K % 16) return fail(NVFP4_ERR_SHAPE, "%s: K=%" PRId64 " is not a multiple of 16", fn, K);
  int64_t wb, sb;
  if (!mul_ok(N, K / 2, &wb) || !mul_ok(N, K / 16, &sb)) return fail(NVFP4_ERR_SHAPE, "%s: N*K overflows", fn);
  if (mo_weight_len != wb)
    return fail(NVFP4_ERR_PLANE, "%s: weight has %" PRId64 " bytes, expected N*K/2 = %" PRId64, fn, mo_weight_len, wb);
  if (mo_weight_scale_len != sb)
    return fail(NVFP4_ERR_PLANE, "%s: weight_scale has %" PRId64 " bytes, expected N*K/16 = %" PRId64, fn,
                mo_weight_scale_len, sb);
  if (!weight_scale_2 || !gs_out) return fail(NVFP4_ERR_NULL, "%s: weight_scale_2 and gs_out are required", fn);
  if (wb > 0 && (!mo_weight || !mo_weight_scale || !w_out || !scales_out))
    return fail(NVFP4_ERR_NULL, "%s: a plane pointer is NULL", fn);
  if (!aligned(mo_weight, 16) || !aligned(mo_weight_scale, 16) || !aligned(w_out, 16) || !aligned(scales_out, 16) ||
      !aligned(weight_scale_2, 4) || !aligned(gs_out, 4))
    return fail(NVFP4_ERR_ALIGN, "%s: planes must be 16-byte aligned, scalars 4-byte", fn);
  return cuda_status(fn, nvfp4::launch_transcode(mo_weight, wb, mo_weight_scale, sb, weight_scale_2, w_out,
                                                 scales_out, gs_out, static_cast<cudaStream_t>(stream)));
}

nvfp4_status nvfp4_transcode_folded(const uint8_t* mo_weight, int64_t mo_weight_len, const uint8_t* mo_weight_scale,
                                    int64_t mo_weight_scale_len, const float* weight_scale_2, int64_t N, int64_t K,
                                    uint32_t* w_out, uint8_t* scales_out, void* stream) {
  const char* fn = "nvfp4_transcode_folded";
  if (N < 0 || K < 0) return fail(NVFP4_ERR_SHAPE, "%s: negative size", fn);
  if (K % 16) return fail(NVFP4_ERR_SHAPE, "%s: K=%" PRId64 " is not a multiple of 16", fn, K);
  int64_t wb, sb;
  if (!mul_ok(N, K / 2, &wb) || !mul_ok(N, K / 16, &sb)) return fail(NVFP4_ERR_SHAPE, "%s: N*K overflows", fn);
  if (mo_weight_len != wb)
    return fail(NVFP4_ERR_PLANE, "%s: weight has %" PRId64 " bytes, expected N*K/2 = %" PRId64, fn, mo_weight_len, wb);
  if (mo_weight_scale_len != sb)
    return fail(NVFP4_ERR_PLANE, "%s: weight_scale has %" PRId64 " bytes, expected N*K/16 = %" PRId64, fn,
                mo_weight_scale_len, sb);
  if (!weight_scale_2) return fail(NVFP4_ERR_NULL, "%s: weight_scale_2 is required", fn);
  if (wb == 0) return ok();
  if (!mo_weight || !mo_weight_scale || !w_out || !scales_out) return fail(NVFP4_ERR_NULL, "%s: a plane pointer is NULL", fn);
  if (!aligned(mo_weight, 16) || !aligned(mo_weight_scale, 16) || !aligned(w_out, 16) || !aligned(scales_out, 16) ||
      !aligned(weight_scale_2, 4))
    return fail(NVFP4_ERR_ALIGN, "%s: planes must be 16-byte aligned, the scalar 4-byte", fn);
  return cuda_status(fn, nvfp4::launch_transcode_folded(mo_weight, wb, mo_weight_scale, sb, weight_scale_2, w_out,
                                                        scales_out, static_cast<cudaStream_t>(stream)));
}

nvfp4_status nvfp4_dequantize(const uint32_t* w, int64_t w_len, const uint8_t* scales, int64_t scales_len,
                              const float* gs, int64_t gs_len, int64_t E, int64_t N, int64_t K,
                              nvfp4_dtype out_dtype, void* out, void* stream) {
  const char* fn = "nvfp4_dequantize";
  if (!dtype_ok(out_dtype)) return fail(NVFP4_ERR_DTYPE, "%s: unknown output dtype %d", fn, (int)out_dtype);
  nvfp4_status s = check_planes(fn, w, w_len, scales, scales_len, E, N, K);
  if (s) return s;
  if ((s = check_gs(fn, gs, gs_len, E))) return s;
  if (w_len == 0) return ok();
  if (!out) return fail(NVFP4_ERR_NULL, "%s: out is NULL", fn);
  if (!aligned(out, 16)) return fail(NVFP4_ERR_ALIGN, "%s: out must be 16-byte aligned", fn);
  return cuda_status(fn, nvfp4::launch_dequantize(w, scales, gs, E, N, K, (int)out_dtype, out,
                                                  static_cast<cudaStream_t>(stream)));
}

nvfp4_status nvfp4_quantize(const void* x, nvfp4_dtype x_dtype, int64_t E, int64_t N, int64_t K, const float* gs,
                            int64_t gs_len, uint32_t* w, int64_t w_len, uint8_t* scales, int64_t scales_len,
                            void* stream) {
  const char* fn = "nvfp4_quantize";
  if (!dtype_ok(x_dtype)) return fail(NVFP4_ERR_DTYPE, "%s: unknown input dtype %d", fn, (int)x_dtype);
  nvfp4_status s = check_planes(fn, w, w_len, scales, scales_len, E, N, K);
  if (s) return s;
  if ((s = check_gs(fn, gs, gs_len, E))) return s;
  if (w_len == 0) return ok();
  if (!x) return fail(NVFP4_ERR_NULL, "%s: x is NULL", fn);
  if (!aligned(x, 16)) return fail(NVFP4_ERR_ALIGN, "%s: x must be 16-byte aligned", fn);
  return cuda_status(fn, nvfp4::launch_quantize(x, (int)x_dtype, gs, E, N, K, w, scales,
                                                static_cast<cudaStream_t>(stream)));
}

int64_t nvfp4_qmm_crossover(nvfp4_dtype x_dtype, int64_t N, int64_t K) {
  const int64_t env = env_crossover();
  if (env >= 0) return env;
  if (x_dtype == NVFP4_F32) return INT64_MAX;  // f32 activations stay on the exact SIMT path
  if (N <= 0 || K <= 0) return kDefaultCrossover;
  // Times in microseconds, fitted to a route sweep (M = 16 .. 256) of the
  // three decode linears on GB300. The decode route (K % 256 == 0) runs one
  // launch per 16 token rows, about 12 + bytes / 3.9 MB each (other K: the
  // cluster kernel, about 8 + bytes / 1.7 MB for the first 16 rows and 0.55
  // of that for each further 16). Below 256 rows the tensor-core route costs
  // one pass of weight decoding over ceil(N / 256) tiles. With the stream-K
  // split that work is spread evenly over the SMs: about 5 + 1.3 us per
  // 64-column k-block of each SM's share (at least 8 k-blocks). Without it,
  // about 0.55 us per k-block while the tiles fit one wave of SMs, 0.8
  // beyond. M* is the first multiple of 16 where the decode route is slower.
  int dev = 0, sms = 152;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    sms = 152;
  const double bytes = 0.5625 * (double)N * (double)K;
  const bool stream = K % 256 == 0;
  const double t16 = stream ? 12.0 + bytes / 3.9e6 : 8.0 + bytes / 1.7e6;
  const int64_t tiles = (N + 255) / 256;
  const double kbs = (double)((K + 63) / 64);
  double t_tc;
  if (nvfp4::tc_stream_k()) {
    const double share = (double)tiles * kbs / sms;
    t_tc = 5.0 + 1.3 * (share > 8.0 ? share : 8.0);
  } else {
    const double waves = (double)((tiles + sms - 1) / sms);
    t_tc = waves * kbs * (tiles <= sms ? 0.55 : 0.8);
  }
  auto t_qmv = [&](int64_t m) {
    const double blocks = (double)((m + 15) / 16);
    return stream ? blocks * t16 : t16 * (1.0 + 0.55 * (blocks - 1.0));
  };
  int64_t m = 16;
  while (m < kDefaultCrossover && t_qmv(m) <= t_tc) m += 16;
  return m;
}

nvfp4_status nvfp4_qmm_routed(const void* x, nvfp4_dtype x_dtype, int64_t M, int64_t K, const uint32_t* w,
                              int64_t w_len, const uint8_t* scales, int64_t scales_len, const float* gs,
                              int64_t gs_len, int64_t N, void* y, nvfp4_route route, void* stream) {
  const char* fn = "nvfp4_qmm";
  if (!dtype_ok(x_dtype)) return fail(NVFP4_ERR_DTYPE, "%s: unknown activation dtype %d", fn, (int)x_dtype);
  if (route != NVFP4_ROUTE_AUTO && route != NVFP4_ROUTE_QMV && route != NVFP4_ROUTE_TC)
    return fail(NVFP4_ERR_DTYPE, "%s: unknown route %d", fn, (int)route);
  if (M < 0) return fail(NVFP4_ERR_SHAPE, "%s: negative M", fn);
  nvfp4_status s = check_planes(fn, w, w_len, scales, scales_len, 1, N, K);
  if (s) return s;
  if ((s = check_gs(fn, gs, gs_len, 1))) return s;
  int64_t xe;
  if (!mul_ok(M, K, &xe) || !mul_ok(M, N, &xe)) return fail(NVFP4_ERR_SHAPE, "%s: M*K or M*N overflows", fn);
  if (M == 0 || N == 0) return ok();
  if (!y || (K > 0 && !x)) return fail(NVFP4_ERR_NULL, "%s: x or y is NULL", fn);
  if (!aligned(x, 16) || !aligned(y, 16)) return fail(NVFP4_ERR_ALIGN, "%s: x and y must be 16-byte aligned", fn);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (K == 0) return cuda_status(fn, cudaMemsetAsync(y, 0, (size_t)(M * N * dtype_size(x_dtype)), st));
  if (route == NVFP4_ROUTE_TC && x_dtype == NVFP4_F32)
    return fail(NVFP4_ERR_DTYPE, "%s: the tensor-core route takes f16 or bf16 activations", fn);
  if (route == NVFP4_ROUTE_TC && !nvfp4::qmm_tc_supported(M, N, K))
    return fail(NVFP4_ERR_SHAPE, "%s: the tensor-core route needs K %% 32 == 0 and K >= 32 (K=%" PRId64 ")", fn, K);
  const bool use_tc = x_dtype != NVFP4_F32 && nvfp4::qmm_tc_supported(M, N, K) &&
                      (route == NVFP4_ROUTE_TC || (route == NVFP4_ROUTE_AUTO && M >= nvfp4_qmm_crossover(x_dtype, N, K)));
  if (use_tc)
    return cuda_status(fn, nvfp4::launch_qmm_tc(x, (int)x_dtype, M, K, w, scales, gs, N, y, st));
  if ((s = check_qmv_grid(fn, M, N))) return s;
  if (x_dtype != NVFP4_F32 && !nvfp4::qmv_supported_k(K))
    return fail(NVFP4_ERR_LIMIT, "%s: K=%" PRId64 " exceeds %" PRId64 " for 16-bit activations", fn, K, nvfp4::kQmvMaxK);
  nvfp4::QmvArgs a{x, w, scales, gs, nullptr, nullptr, M, M, K, N, 1, y};
  return cuda_status(fn, run_qmv(a, (int)x_dtype, st));
}

nvfp4_status nvfp4_qmm(const void* x, nvfp4_dtype x_dtype, int64_t M, int64_t K, const uint32_t* w,
                       int64_t w_len, const uint8_t* scales, int64_t scales_len, const float* gs,
                       int64_t gs_len, int64_t N, void* y, void* stream) {
  return nvfp4_qmm_routed(x, x_dtype, M, K, w, w_len, scales, scales_len, gs, gs_len, N, y, NVFP4_ROUTE_AUTO,
                          stream);
}

nvfp4_status nvfp4_qmm_glu(const void* x, nvfp4_dtype x_dtype, int64_t M, int64_t K, const uint32_t* w,
                           int64_t w_len, const uint8_t* scales, int64_t scales_len, const float* gs,
                           int64_t gs_len, int64_t I, nvfp4_act act, void* y, nvfp4_route route, void* stream) {
  const char* fn = "nvfp4_qmm_glu";
  if (x_dtype != NVFP4_F16 && x_dtype != NVFP4_BF16)
    return fail(NVFP4_ERR_DTYPE, "%s: f16 or bf16 activations only (got %d)", fn, (int)x_dtype);
  if (act != NVFP4_ACT_SILU && act != NVFP4_ACT_GELU_TANH)
    return fail(NVFP4_ERR_DTYPE, "%s: unknown activation %d", fn, (int)act);
  if (route != NVFP4_ROUTE_AUTO && route != NVFP4_ROUTE_QMV && route != NVFP4_ROUTE_TC)
    return fail(NVFP4_ERR_DTYPE, "%s: unknown route %d", fn, (int)route);
  if (M < 0 || I < 0) return fail(NVFP4_ERR_SHAPE, "%s: negative M or I", fn);
  if (I > (INT64_MAX >> 2)) return fail(NVFP4_ERR_SHAPE, "%s: I too large", fn);
  const int64_t N = 2 * I;  // gate rows, then up rows
  nvfp4_status s = check_planes(fn, w, w_len, scales, scales_len, 1, N, K);
  if (s) return s;
  if ((s = check_gs(fn, gs, gs_len, 1))) return s;
  int64_t xe;
  if (!mul_ok(M, K, &xe) || !mul_ok(M, N, &xe)) return fail(NVFP4_ERR_SHAPE, "%s: M*K or M*N overflows", fn);
  if (M == 0 || I == 0) return ok();
  if (!y || (K > 0 && !x)) return fail(NVFP4_ERR_NULL, "%s: x or y is NULL", fn);
  if (!aligned(x, 16) || !aligned(y, 16)) return fail(NVFP4_ERR_ALIGN, "%s: x and y must be 16-byte aligned", fn);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // K = 0: both halves are 0 and so is act(0) * 0
  if (K == 0) return cuda_status(fn, cudaMemsetAsync(y, 0, (size_t)(M * I * dtype_size(x_dtype)), st));
  const bool tc_ok = nvfp4::qmm_tc_supported(M, N, K);
  nvfp4::QmvArgs a{x, w, scales, gs, nullptr, nullptr, M, M, K, N, 1, y};
  a.glu_cols = I;
  a.glu_act = (int)act;
  const bool qmv_ok = nvfp4::qmv_stream_supported(a, (int)x_dtype) && N < (1ll << 31);
  bool use_tc;
  if (route == NVFP4_ROUTE_TC)
    use_tc = true;
  else if (route == NVFP4_ROUTE_QMV)
    use_tc = false;
  else
    use_tc = !qmv_ok || M >= nvfp4_qmm_crossover(x_dtype, N, K);
  if (use_tc && !tc_ok)
    return fail(NVFP4_ERR_SHAPE, "%s: the tensor-core route needs K %% 32 == 0 and K >= 32 (K=%" PRId64 ")", fn, K);
  if (!use_tc && !qmv_ok)
    return fail(NVFP4_ERR_SHAPE, "%s: the decode route needs K %% 256 == 0 (K=%" PRId64 ")", fn, K);
  if (use_tc) return cuda_status(fn, nvfp4::launch_qmm_tc_glu(x, (int)x_dtype, M, K, w, scales, gs, I, (int)act, y, st));
  return cuda_status(fn, nvfp4::launch_qmv_stream_glu(a, (int)x_dtype, st));
}

nvfp4_status nvfp4_qmm_nontransposed(const void* x, nvfp4_dtype x_dtype, int64_t M, int64_t K, const uint32_t* w,
                                     int64_t w_len, const uint8_t* scales, int64_t scales_len, const float* gs,
                                     int64_t gs_len, int64_t N, void* y, void* stream) {
  const char* fn = "nvfp4_qmm_nontransposed";
  if (x_dtype != NVFP4_F16 && x_dtype != NVFP4_BF16)
    return fail(NVFP4_ERR_DTYPE, "%s: f16 or bf16 activations only (got %d)", fn, (int)x_dtype);
  if (M < 0 || K < 0 || N < 0) return fail(NVFP4_ERR_SHAPE, "%s: negative size", fn);
  // the quantized axis of a non-transposed plane is N
  if (N % 16) return fail(NVFP4_ERR_SHAPE, "%s: N=%" PRId64 " (the quantized axis) is not a multiple of 16", fn, N);
  nvfp4_status s = check_planes(fn, w, w_len, scales, scales_len, 1, K, N);  // [K, N/8] words, [K, N/16] scales
  if (s) return s;
  if ((s = check_gs(fn, gs, gs_len, 1))) return s;
  int64_t xe;
  if (!mul_ok(M, K, &xe) || !mul_ok(M, N, &xe)) return fail(NVFP4_ERR_SHAPE, "%s: M*K or M*N overflows", fn);
  if (M == 0 || N == 0) return ok();
  if (!y || (K > 0 && !x)) return fail(NVFP4_ERR_NULL, "%s: x or y is NULL", fn);
  if (!aligned(x, 16) || !aligned(y, 16)) return fail(NVFP4_ERR_ALIGN, "%s: x and y must be 16-byte aligned", fn);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (K == 0) return cuda_status(fn, cudaMemsetAsync(y, 0, (size_t)(M * N * dtype_size(x_dtype)), st));
  // up to sixteen token rows: streaming passes (the NVFP4_OPT_NT_DECODE option
  // set to 0 sends every M to the tensor cores)
  if (nvfp4::option(nvfp4::kOptNtDecode) != 0 && nvfp4::qmv_nt_supported(M, N, K))
    return cuda_status(fn, nvfp4::launch_qmv_nt(x, (int)x_dtype, M, K, w, scales, gs, N, y, st));
  if (!nvfp4::qmm_tc_nt_supported(M, N, K))
    return fail(NVFP4_ERR_LIMIT, "%s: M or K of 2^31 or more, or too many tiles", fn);
  return cuda_status(fn, nvfp4::launch_qmm_tc_nt(x, (int)x_dtype, M, K, w, scales, gs, N, y, st));
}

nvfp4_status nvfp4_qmm_batched(const void* x, nvfp4_dtype x_dtype, int64_t batches, int64_t M, int64_t K,
                               const uint32_t* w, int64_t w_len, const uint8_t* scales, int64_t scales_len,
                               const float* gs, int64_t gs_len, int64_t N, void* y, void* stream) {
  const char* fn = "nvfp4_qmm_batched";
  if (!dtype_ok(x_dtype)) return fail(NVFP4_ERR_DTYPE, "%s: unknown activation dtype %d", fn, (int)x_dtype);
  if (batches < 0 || M < 0) return fail(NVFP4_ERR_SHAPE, "%s: negative batch count or M", fn);
  nvfp4_status s = check_planes(fn, w, w_len, scales, scales_len, batches, N, K);
  if (s) return s;
  if ((s = check_gs(fn, gs, gs_len, batches))) return s;
  int64_t rows, xe;
  if (!mul_ok(batches, M, &rows) || !mul_ok(rows, K, &xe) || !mul_ok(rows, N, &xe))
    return fail(NVFP4_ERR_SHAPE, "%s: batches*M*K or batches*M*N overflows", fn);
  if (rows == 0 || N == 0) return ok();
  if (!y || (K > 0 && !x)) return fail(NVFP4_ERR_NULL, "%s: x or y is NULL", fn);
  if (!aligned(x, 16) || !aligned(y, 16)) return fail(NVFP4_ERR_ALIGN, "%s: x and y must be 16-byte aligned", fn);
  if (batches > INT32_MAX) return fail(NVFP4_ERR_LIMIT, "%s: more than 2^31-1 batches", fn);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (K == 0) return cuda_status(fn, cudaMemsetAsync(y, 0, (size_t)(rows * N * dtype_size(x_dtype)), st));
  // Decode-size batches go out as one launch of the expert-group route: row
  // r of the flattened [batches * M, K] activations uses batch r / M's plane.
  if (x_dtype != NVFP4_F32 && M < nvfp4_qmm_crossover(x_dtype, N, K)) {
    nvfp4::QmvArgs a{x, w, scales, gs, nullptr, nullptr, rows, rows, K, N, batches, y};
    a.rows_per_expert = M;
    if (nvfp4::qmv_group_supported(a, (int)x_dtype)) return cuda_status(fn, nvfp4::launch_qmv_group(a, (int)x_dtype, st));
  }
  // Otherwise one QuantizedMatmul per batch, each on its own route.
  const int64_t xs = dtype_size(x_dtype);
  for (int64_t b = 0; b < batches; ++b) {
    s = nvfp4_qmm(static_cast<const char*>(x) + b * M * K * xs, x_dtype, M, K, w + b * N * (K / 8), N * (K / 8),
                  scales + b * N * (K / 16), N * (K / 16), gs ? gs + b : nullptr, gs ? 1 : 0, N,
                  static_cast<char*>(y) + b * M * N * xs, stream);
    if (s) return s;
  }
  return ok();
}

nvfp4_status nvfp4_qmm_noalloc(const void* x, nvfp4_dtype x_dtype, int64_t M, int64_t K, const uint32_t* w,
                               int64_t w_len, const uint8_t* scales, int64_t scales_len, const float* gs,
                               int64_t gs_len, int64_t N, void* y, void* stream) {
  const char* fn = "nvfp4_qmm_noalloc";
  if (x_dtype != NVFP4_F16 && x_dtype != NVFP4_BF16)
    return fail(NVFP4_ERR_DTYPE, "%s: takes f16 or bf16 activations (dtype %d)", fn, (int)x_dtype);
  if (M < 0) return fail(NVFP4_ERR_SHAPE, "%s: negative M", fn);
  nvfp4_status s = check_planes(fn, w, w_len, scales, scales_len, 1, N, K);
  if (s) return s;
  if ((s = check_gs(fn, gs, gs_len, 1))) return s;
  int64_t xe;
  if (!mul_ok(M, K, &xe) || !mul_ok(M, N, &xe)) return fail(NVFP4_ERR_SHAPE, "%s: M*K or M*N overflows", fn);
  if (M == 0 || N == 0) return ok();
  if (!y || (K > 0 && !x)) return fail(NVFP4_ERR_NULL, "%s: x or y is NULL", fn);
  if (!aligned(x, 16) || !aligned(y, 16)) return fail(NVFP4_ERR_ALIGN, "%s: x and y must be 16-byte aligned", fn);
  if (M > 16) return fail(NVFP4_ERR_LIMIT, "%s: M=%" PRId64 " exceeds 16 token rows", fn, M);
  if (K % 256) return fail(NVFP4_ERR_SHAPE, "%s: K=%" PRId64 " is not a multiple of 256", fn, K);
  if (K > (int64_t)1 << 20) return fail(NVFP4_ERR_LIMIT, "%s: K=%" PRId64 " exceeds 2^20", fn, K);
  if (N > nvfp4::kNoAllocMaxRows)
    return fail(NVFP4_ERR_LIMIT, "%s: N=%" PRId64 " exceeds the %" PRId64 " weight rows its fixed scratch covers", fn, N,
                nvfp4::kNoAllocMaxRows);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (K == 0) return cuda_status(fn, cudaMemsetAsync(y, 0, (size_t)(M * N * dtype_size(x_dtype)), st));
  nvfp4::QmvArgs a{x, w, scales, gs, nullptr, nullptr, M, M, K, N, 1, y};
  const cudaError_t e = nvfp4::launch_qmv_stream_noalloc(a, (int)x_dtype, st);
  if (e == cudaErrorInvalidConfiguration)
    return fail(NVFP4_ERR_LIMIT, "%s: no launch plan of the decode kernel fits this shape (N=%" PRId64 ", K=%" PRId64
                ", M=%" PRId64 ")", fn, N, K, M);
  return cuda_status(fn, e);
}

nvfp4_status nvfp4_qmm_sequence(const nvfp4_qmm_call* calls, int32_t ncalls, nvfp4_dtype x_dtype, void* stream) {
  const char* fn = "nvfp4_qmm_sequence";
  if (x_dtype != NVFP4_F16 && x_dtype != NVFP4_BF16)
    return fail(NVFP4_ERR_DTYPE, "%s: takes f16 or bf16 activations (dtype %d)", fn, (int)x_dtype);
  if (ncalls < 0 || ncalls > nvfp4::kSeqMaxCallsApi)
    return fail(NVFP4_ERR_LIMIT, "%s: ncalls=%d outside 0..%d", fn, (int)ncalls, nvfp4::kSeqMaxCallsApi);
  if (ncalls > 0 && !calls) return fail(NVFP4_ERR_NULL, "%s: calls is NULL", fn);
  nvfp4::QmvArgs args[nvfp4::kSeqMaxCallsApi];
  int deps[nvfp4::kSeqMaxCallsApi];
  int n = 0;
  char name[64];
  for (int32_t c = 0; c < ncalls; ++c) {
    const nvfp4_qmm_call& q = calls[c];
    snprintf(name, sizeof(name), "%s: call %d", fn, (int)c);
    if (q.M < 0) return fail(NVFP4_ERR_SHAPE, "%s: negative M", name);
    nvfp4_status s = check_planes(name, q.w, q.w_len, q.scales, q.scales_len, 1, q.N, q.K);
    if (s) return s;
    if ((s = check_gs(name, q.gs, q.gs_len, 1))) return s;
    int64_t xe;
    if (!mul_ok(q.M, q.K, &xe) || !mul_ok(q.M, q.N, &xe)) return fail(NVFP4_ERR_SHAPE, "%s: M*K or M*N overflows", name);
    if (q.M == 0 || q.N == 0) continue;  // empty output: nothing to run
    if (!q.y || !q.x) return fail(NVFP4_ERR_NULL, "%s: x or y is NULL", name);
    if (!aligned(q.x, 16) || !aligned(q.y, 16))
      return fail(NVFP4_ERR_ALIGN, "%s: x and y must be 16-byte aligned", name);
    if (q.M > 16) return fail(NVFP4_ERR_LIMIT, "%s: M=%" PRId64 " exceeds 16 token rows", name, q.M);
    if (q.K == 0 || q.K % 256)
      return fail(NVFP4_ERR_SHAPE, "%s: K=%" PRId64 " is not a positive multiple of 256", name, q.K);
    if (q.K > (int64_t)1 << 20) return fail(NVFP4_ERR_LIMIT, "%s: K=%" PRId64 " exceeds 2^20", name, q.K);
    if (q.N >= ((int64_t)1 << 31)) return fail(NVFP4_ERR_LIMIT, "%s: N=%" PRId64 " exceeds 2^31-1", name, q.N);
    args[n] = nvfp4::QmvArgs{q.x, q.w, q.scales, q.gs, nullptr, nullptr, q.M, q.M, q.K, q.N, 1, q.y};
    // a call whose predecessors were all empty has nothing to wait for
    deps[n] = n > 0 && q.after_previous != 0 ? 1 : 0;
    ++n;
  }
  if (n == 0) return ok();
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const cudaError_t e = nvfp4::launch_qmv_seq(args, deps, n, (int)x_dtype, st);
  if (e == cudaErrorInvalidConfiguration)
    return fail(NVFP4_ERR_LIMIT, "%s: no launch plan of the decode kernel fits these %d calls", fn, n);
  return cuda_status(fn, e);
}

nvfp4_status nvfp4_gather_qmm(const void* x, nvfp4_dtype x_dtype, int64_t B, int64_t K, const uint32_t* lhs_indices,
                              const uint32_t* rhs_indices, int64_t R, int sorted_indices, const uint32_t* w,
                              int64_t w_len, const uint8_t* scales, int64_t scales_len, const float* gs,
                              int64_t gs_len, int64_t E, int64_t N, void* y, void* stream) {
  const char* fn = "nvfp4_gather_qmm";
  if (!dtype_ok(x_dtype)) return fail(NVFP4_ERR_DTYPE, "%s: unknown activation dtype %d", fn, (int)x_dtype);
  if (B < 0 || R < 0) return fail(NVFP4_ERR_SHAPE, "%s: negative B or R", fn);
  nvfp4_status s = check_planes(fn, w, w_len, scales, scales_len, E, N, K);
  if (s) return s;
  if ((s = check_gs(fn, gs, gs_len, E))) return s;
  int64_t xe;
  if (!mul_ok(B, K, &xe) || !mul_ok(R, N, &xe)) return fail(NVFP4_ERR_SHAPE, "%s: B*K or R*N overflows", fn);
  if (R == 0 || N == 0) return ok();
  if (!y || !rhs_indices) return fail(NVFP4_ERR_NULL, "%s: y and rhs_indices are required", fn);
  if (B > 0 && K > 0 && !x) return fail(NVFP4_ERR_NULL, "%s: x is NULL", fn);
  if (!aligned(x, 16) || !aligned(y, 16)) return fail(NVFP4_ERR_ALIGN, "%s: x and y must be 16-byte aligned", fn);
  if (!aligned(rhs_indices, 4) || !aligned(lhs_indices, 4))
    return fail(NVFP4_ERR_ALIGN, "%s: index arrays must be 4-byte aligned", fn);
  if ((s = check_qmv_grid(fn, R, N))) return s;
  if (x_dtype != NVFP4_F32 && !nvfp4::qmv_supported_k(K))
    return fail(NVFP4_ERR_LIMIT, "%s: K=%" PRId64 " exceeds %" PRId64 " for 16-bit activations", fn, K, nvfp4::kQmvMaxK);
  if (E > INT32_MAX) return fail(NVFP4_ERR_LIMIT, "%s: E=%" PRId64 " exceeds 2^31-1", fn, E);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (K == 0) return cuda_status(fn, cudaMemsetAsync(y, 0, (size_t)(R * N * dtype_size(x_dtype)), st));
  // Sorted rows with enough of them per expert take the expert-batched
  // tensor-core route (128-row tiles; below about 16 rows per expert the tiles
  // would mostly be padding). The NVFP4_OPT_GATHER_TC option forces (1) or
  // disables (0) it.
  if (sorted_indices && x_dtype != NVFP4_F32 && nvfp4::gather_tc_supported(B, K, R, E, N)) {
    const int force = nvfp4::option(nvfp4::kOptGatherTc);
    const bool use = force >= 0 ? force == 1 : (R >= 512 && R >= 16 * E);
    if (use)
      return cuda_status(fn, nvfp4::launch_gather_tc(x, (int)x_dtype, B, K, lhs_indices, rhs_indices, R, w, scales, gs,
                                                     E, N, y, st));
  }
  nvfp4::QmvArgs a{x, w, scales, gs, lhs_indices, rhs_indices, B, R, K, N, E, y};
  return cuda_status(fn, run_qmv(a, (int)x_dtype, st));
}

}  // extern "C"
