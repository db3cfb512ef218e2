// Decode-size QuantizedMatmul with a non-transposed weight (mlx PR #2629,
// Changes during review: the quantized axis of such a weight is N): y = x @
// dequantize(w) * gs / 2688 for one or two token rows, w [K, N/8] words
// (word j of row k holds outputs 8j..8j+7 of input k), one E4M3 byte per 16
// outputs of an input.
//
// The weight plane is streamed once. A warp task is 32 word columns (256
// outputs) by 128 inputs: lane j decodes word column j of each input row (a
// warp load is 128 contiguous bytes of one row), multiplies the eight exact
// products fp4 * e4m3 by the row's activations (loaded with the words, one
// broadcast request per token row and eight inputs) and keeps eight float
// sums per token row. Tasks split K, so each task adds its sums into a float
// workspace [M, N] (red.global.add); a second kernel scales, rounds and
// writes y, and returns the workspace to zero for the next call.
#include <cstdint>
#include <map>
#include <mutex>
#include <vector>

#include "nvfp4_common.cuh"
#include "nvfp4_internal.h"

namespace nvfp4 {

namespace {

constexpr int kNtThreads = 256;  // eight warps
constexpr int kNtWarps = kNtThreads / 32;
constexpr int kNtChunk = 128;    // inputs per task (a multiple of 16)

// Eight input rows of the lane's word column, the token rows' activations
// at those inputs (raw, eight 16-bit values per token row) and, per lane, one
// word of scale bytes: bytes 4 (lane & 3) .. + 3 of the task's 16 for input
// row lane / 4. Loads only, so a later group's loads never wait on this one's.
template <int MT>
struct NtGroup {
  uint32_t w[8];
  uint32_t s;
  uint4 x[MT];
};

template <typename T, int MT>
__device__ __forceinline__ void nt_load(NtGroup<MT>& g, const T* __restrict__ x, int M, int64_t K,
                                        const uint32_t* __restrict__ w, const uint8_t* __restrict__ scales,
                                        int64_t nwords, int64_t ngroups, int64_t col, bool cok, int64_t k, int rows,
                                        int64_t g0, int lane) {
#pragma unroll
  for (int kk = 0; kk < 8; ++kk) g.w[kk] = cok && kk < rows ? __ldg(w + (k + kk) * nwords + col) : 0u;
  uint32_t sv = 0;
  const int r = lane >> 2;
  if (r < rows) {
    const uint8_t* row = scales + (k + r) * ngroups;
    if ((ngroups & 3) == 0) {
      if (g0 < ngroups) sv = __ldg(reinterpret_cast<const uint32_t*>(row + g0));
    } else {
      for (int q = 0; q < 4; ++q)
        if (g0 + q < ngroups) sv |= (uint32_t)__ldg(row + g0 + q) << (8 * q);
    }
  }
  g.s = sv;
  // every lane loads the same activations (one broadcast request a row)
  const bool vec = rows >= 8 && (K & 7) == 0;
#pragma unroll
  for (int m = 0; m < MT; ++m) {
    if (m < M && vec) {
      g.x[m] = __ldg(reinterpret_cast<const uint4*>(x + (int64_t)m * K + k));
    } else {
      uint16_t h[8];
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
        h[kk] = m < M && kk < rows ? __ldg(reinterpret_cast<const unsigned short*>(x) + (int64_t)m * K + k + kk) : 0;
      g.x[m] = make_uint4(h[0] | ((uint32_t)h[1] << 16), h[2] | ((uint32_t)h[3] << 16), h[4] | ((uint32_t)h[5] << 16),
                          h[6] | ((uint32_t)h[7] << 16));
    }
  }
}

// Activation kk of a row's eight, as f32.
template <typename T> __device__ __forceinline__ float x_at(const uint4& v, int kk);
template <> __device__ __forceinline__ float x_at<__nv_bfloat16>(const uint4& v, int kk) {
  const uint32_t u = kk < 2 ? v.x : kk < 4 ? v.y : kk < 6 ? v.z : v.w;
  return __uint_as_float((kk & 1) ? (u & 0xFFFF0000u) : (u << 16));
}
template <> __device__ __forceinline__ float x_at<__half>(const uint4& v, int kk) {
  const uint32_t u = kk < 2 ? v.x : kk < 4 ? v.y : kk < 6 ? v.z : v.w;
  return __half2float(__ushort_as_half((unsigned short)((kk & 1) ? (u >> 16) : (u & 0xFFFFu))));
}

// (c0, c1) += (a, a) * (b0, b1), each an IEEE fma (one packed instruction).
__device__ __forceinline__ void fma2(float& c0, float& c1, float a, float b0, float b1) {
  asm("{\n\t.reg .b64 pa, pb, pc;\n\t"
      "mov.b64 pa, {%2, %2};\n\t"
      "mov.b64 pb, {%3, %4};\n\t"
      "mov.b64 pc, {%0, %1};\n\t"
      "fma.rn.f32x2 pc, pa, pb, pc;\n\t"
      "mov.b64 {%0, %1}, pc;\n\t}"
      : "+f"(c0), "+f"(c1)
      : "f"(a), "f"(b0), "f"(b1));
}

// The block scale goes into the activation (x * e4m3 has at most 15
// significant bits, exact in f32), so each code needs only its E2M1 value;
// every product x * e4m3 * fp4 is exact as before.
template <typename T, int MT>
__device__ __forceinline__ void nt_accumulate(const NtGroup<MT>& g, int lane, float (&acc)[MT][8]) {
#pragma unroll
  for (int kk = 0; kk < 8; ++kk) {
    const uint32_t quad = __shfl_sync(0xffffffffu, g.s, kk * 4 + (lane >> 3));
    const float sf = e4m3_to_f32((quad >> (8 * ((lane >> 1) & 3))) & 0xFFu);
    uint32_t h[4];
    e2m1x8_to_f16x2(g.w[kk], h);
    float v[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h[i]));
      v[2 * i] = f.x;
      v[2 * i + 1] = f.y;
    }
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      const float xs = __fmul_rn(x_at<T>(g.x[m], kk), sf);
#pragma unroll
      for (int i = 0; i < 4; ++i) fma2(acc[m][2 * i], acc[m][2 * i + 1], xs, v[2 * i], v[2 * i + 1]);
    }
  }
}

template <typename T, int MT>
__global__ void __launch_bounds__(kNtThreads)
qmv_nt_kernel(const T* __restrict__ x, int M, int64_t K, const uint32_t* __restrict__ w,
              const uint8_t* __restrict__ scales, int64_t N, float* __restrict__ ws, int64_t slabs, int64_t tasks) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t nwords = N / 8, ngroups = N / 16;
  const int64_t nw = (int64_t)gridDim.x * kNtWarps;
  for (int64_t t = (int64_t)blockIdx.x * kNtWarps + warp; t < tasks; t += nw) {  // warp-uniform
    const int64_t slab = t % slabs, k0 = (t / slabs) * kNtChunk;
    const int kn = (int)(K - k0 < kNtChunk ? K - k0 : kNtChunk);
    const int64_t col = slab * 32 + lane, g0 = slab * 16 + 4 * (lane & 3);
    const bool cok = col < nwords;
    float acc[MT][8];
#pragma unroll
    for (int m = 0; m < MT; ++m)
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[m][i] = 0.0f;
    // two groups of eight rows in flight: the next group's loads are issued
    // before the current group is decoded
    NtGroup<MT> ga, gb;
    nt_load<T, MT>(ga, x, M, K, w, scales, nwords, ngroups, col, cok, k0, kn, g0, lane);
    for (int kb = 0; kb < kn; kb += 16) {
      nt_load<T, MT>(gb, x, M, K, w, scales, nwords, ngroups, col, cok, k0 + kb + 8, kn - kb - 8, g0, lane);
      nt_accumulate<T, MT>(ga, lane, acc);
      if (kb + 16 < kn) nt_load<T, MT>(ga, x, M, K, w, scales, nwords, ngroups, col, cok, k0 + kb + 16, kn - kb - 16, g0, lane);
      if (kb + 8 < kn) nt_accumulate<T, MT>(gb, lane, acc);
    }
    if (cok) {
#pragma unroll
      for (int m = 0; m < MT; ++m) {
        if (m >= M) break;
        float* dst = ws + (int64_t)m * N + col * 8;
#pragma unroll
        for (int i = 0; i < 8; ++i) atomicAdd(dst + i, acc[m][i]);
      }
    }
  }
}

// y = cast(ws * gs / 2688); the workspace returns to zero.
template <typename T>
__global__ void __launch_bounds__(256) qmv_nt_finish(float* __restrict__ ws, int64_t n, const float* __restrict__ gs,
                                                     T* __restrict__ y) {
  const float fac = global_factor(gs, 0);
  const bool has_gs = gs != nullptr;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
    const float v = ws[i];
    ws[i] = 0.0f;
    y[i] = from_f32<T>(has_gs ? __fmul_rn(v, fac) : v);
  }
}

// Float workspace [kQmvNtMaxM, N] per (device, stream), zero when handed
// out; grown on demand (a new buffer is zeroed on the calling stream, so a
// captured call zeroes it in every replay) and kept until
// release_nt_workspaces().
std::mutex g_nt_mu;
std::map<std::pair<int, uintptr_t>, std::pair<float*, size_t>> g_nt;
std::vector<float*> g_nt_retired;

cudaError_t nt_workspace(int dev, cudaStream_t st, size_t floats, float** out) {
  std::lock_guard<std::mutex> lock(g_nt_mu);
  auto& slot = g_nt[{dev, reinterpret_cast<uintptr_t>(st)}];
  if (slot.second < floats) {
    cudaStreamCaptureMode mode = cudaStreamCaptureModeRelaxed;
    cudaError_t e = cudaThreadExchangeStreamCaptureMode(&mode);
    if (e != cudaSuccess) return e;
    float* ptr = nullptr;
    e = cudaMalloc(&ptr, floats * sizeof(float));
    cudaStreamCaptureMode back = mode;
    cudaThreadExchangeStreamCaptureMode(&back);
    if (e != cudaSuccess) return e;
    if ((e = cudaMemsetAsync(ptr, 0, floats * sizeof(float), st)) != cudaSuccess) return e;
    if (slot.first) g_nt_retired.push_back(slot.first);
    slot = {ptr, floats};
  }
  *out = slot.first;
  return cudaSuccess;
}

template <typename T, int MT>
cudaError_t launch_mt(const void* x, int64_t M, int64_t K, const uint32_t* w, const uint8_t* scales, const float* gs,
                      int64_t N, void* y, float* ws, int sms, cudaStream_t st) {
  const int64_t slabs = (N / 8 + 31) / 32, tasks = slabs * ((K + kNtChunk - 1) / kNtChunk);
  int per_sm = 1;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, qmv_nt_kernel<T, MT>, kNtThreads, 0) != cudaSuccess ||
      per_sm < 1)
    per_sm = 1;
  const int64_t want = (tasks + kNtWarps - 1) / kNtWarps, cap = (int64_t)sms * per_sm;
  qmv_nt_kernel<T, MT><<<(unsigned)(want < cap ? want : cap), kNtThreads, 0, st>>>(
      static_cast<const T*>(x), (int)M, K, w, scales, N, ws, slabs, tasks);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int64_t n = M * N, fb = (n + 255) / 256;
  qmv_nt_finish<T><<<(unsigned)(fb < 4 * sms ? fb : 4 * sms), 256, 0, st>>>(ws, n, gs, static_cast<T*>(y));
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_t(const void* x, int64_t M, int64_t K, const uint32_t* w, const uint8_t* scales, const float* gs,
                     int64_t N, void* y, cudaStream_t st) {
  int dev = 0, sms = 152;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  float* ws = nullptr;
  cudaError_t e = nt_workspace(dev, st, (size_t)kQmvNtMaxM * (size_t)N, &ws);
  if (e != cudaSuccess) return e;
  if (M == 1) return launch_mt<T, 1>(x, M, K, w, scales, gs, N, y, ws, sms, st);
  return launch_mt<T, 2>(x, M, K, w, scales, gs, N, y, ws, sms, st);
}

}  // namespace

bool qmv_nt_supported(int64_t M, int64_t N, int64_t K) {
  return M >= 1 && M <= kQmvNtMaxM && N > 0 && N % 16 == 0 && K > 0 && N < (1ll << 40) && K < (1ll << 40);
}

cudaError_t launch_qmv_nt(const void* x, int xdt, int64_t M, int64_t K, const uint32_t* w, const uint8_t* scales,
                          const float* gs, int64_t N, void* y, cudaStream_t st) {
  if (xdt == kBF16) return launch_t<__nv_bfloat16>(x, M, K, w, scales, gs, N, y, st);
  return launch_t<__half>(x, M, K, w, scales, gs, N, y, st);
}

void release_nt_workspaces() {
  std::lock_guard<std::mutex> lock(g_nt_mu);
  for (auto& kv : g_nt) cudaFree(kv.second.first);
  g_nt.clear();
  for (float* p : g_nt_retired) cudaFree(p);
  g_nt_retired.clear();
}

}  // namespace nvfp4
