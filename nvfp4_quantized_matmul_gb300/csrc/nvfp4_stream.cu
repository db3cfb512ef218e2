// Bandwidth-bound kernels: ModelOpt-triplet transcode and exact dequantize.
#include <cstdlib>

#include "nvfp4_common.cuh"
#include "nvfp4_internal.h"
#include "nvfp4_pipe.cuh"

namespace nvfp4 {

__device__ int g_copy_error = 0;  // first error code recorded by a bounded wait of the bulk copy

namespace {

constexpr int kStreamThreads = 256;

// Grid for a grid-stride kernel: enough blocks for `units` thread-iterations,
// at most what is resident at once (a second wave of equal blocks would run
// after the first instead of beside it).
template <typename Kern>
int stream_grid(Kern kern, int64_t units) {
  int dev = 0, sms = 152, per_sm = 1;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kStreamThreads, 0) != cudaSuccess || per_sm < 1)
    per_sm = 1;
  const int64_t want = (units + kStreamThreads - 1) / kStreamThreads;
  const int64_t cap = (int64_t)sms * per_sm;
  return (int)(want < cap ? (want < 1 ? 1 : want) : cap);
}

// Transcode (issue #693 "direct-transcode ModelOpt triplets to MLX native",
// Implementation plan step 3). ModelOpt's U8 plane stores column 2j in the
// low nibble of byte j; packing four consecutive bytes little-endian into one
// uint32 therefore yields the native word with column 8i+k in nibble k. That
// repack is the identity on the byte stream, so the kernel copies both planes
// as they are; the E4M3 block scales are kept byte for byte and the sidecar is
// f32(ws2) * 2688 so that gs / 2688 stands for ws2. Both planes are read and
// written exactly once; no dense intermediate.
//
// The copy engine moves the bytes: each CTA (one per SM, one thread issuing)
// copies a contiguous run of 32 KB chunks of both planes through a ring of
// six shared-memory buffers, bulk loads running up to six chunks ahead of the
// bulk stores, a handful of instructions per 32 KB (a 16-byte vector copy
// with eight loads in flight per thread took 80 us for a layer's three
// triplets, this one 75). Sizes and addresses of bulk copies must be
// multiples of 16 bytes: the last (< 16) bytes of each plane are copied by
// plain stores.
constexpr uint32_t kCopyChunk = 32 * 1024;
constexpr int kCopyBufs = 6;

__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}
__device__ __forceinline__ void bulk_s2g(void* dst, uint32_t src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(src), "r"(bytes)
               : "memory");
}

__global__ void __launch_bounds__(32, 1)
transcode_bulk_kernel(const uint8_t* __restrict__ mo_w, int64_t w_bytes, const uint8_t* __restrict__ mo_ws,
                      int64_t s_bytes, const float* __restrict__ ws2, uint8_t* __restrict__ w_out,
                      uint8_t* __restrict__ s_out, float* __restrict__ gs_out) {
  extern __shared__ __align__(128) uint8_t buf[];
  __shared__ __align__(8) uint64_t bars[kCopyBufs];
  __shared__ int abort_flag;
  const int64_t wv = w_bytes & ~(int64_t)15, sv = s_bytes & ~(int64_t)15;
  const int64_t n0 = (wv + kCopyChunk - 1) / kCopyChunk, n = n0 + (sv + kCopyChunk - 1) / kCopyChunk;
  if (blockIdx.x == 0) {
    if (threadIdx.x == 0) gs_out[0] = __fmul_rn(__ldg(ws2), kGlobalScaleDivisor);
    if (threadIdx.x < w_bytes - wv) w_out[wv + threadIdx.x] = mo_w[wv + threadIdx.x];
    if (threadIdx.x < s_bytes - sv) s_out[sv + threadIdx.x] = mo_ws[sv + threadIdx.x];
  }
  if (threadIdx.x != 0) return;
  // chunk c: source, destination and size
  auto chunk = [&](int64_t c, const uint8_t*& src, uint8_t*& dst, uint32_t& bytes) {
    if (c < n0) {
      const int64_t off = c * kCopyChunk;
      src = mo_w + off;
      dst = w_out + off;
      bytes = (uint32_t)(wv - off < kCopyChunk ? wv - off : kCopyChunk);
    } else {
      const int64_t off = (c - n0) * kCopyChunk;
      src = mo_ws + off;
      dst = s_out + off;
      bytes = (uint32_t)(sv - off < kCopyChunk ? sv - off : kCopyChunk);
    }
  };
  const int64_t c0 = n * blockIdx.x / gridDim.x, c1 = n * (blockIdx.x + 1) / gridDim.x;
  const uint32_t sbuf = pipe::smem_addr(buf), sbar = pipe::smem_addr(bars);
  abort_flag = 0;
  for (int k = 0; k < kCopyBufs; ++k) pipe::mbar_init(sbar + 8u * k, 1);
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  int64_t issued = c0;  // next chunk to load
  for (; issued < c1 && issued < c0 + kCopyBufs; ++issued) {
    const uint8_t* src;
    uint8_t* dst;
    uint32_t bytes;
    chunk(issued, src, dst, bytes);
    const int k = (int)(issued - c0);
    pipe::mbar_arrive_tx(sbar + 8u * k, bytes);
    bulk_g2s(sbuf + (uint32_t)k * kCopyChunk, src, bytes, sbar + 8u * k);
  }
  int64_t i = c0;
  for (; i < c1; ++i) {
    const int k = (int)((i - c0) % kCopyBufs);
    const uint32_t ph = (uint32_t)(((i - c0) / kCopyBufs) & 1);
    if (!pipe::wait_bar(sbar + 8u * k, ph, &abort_flag, 41, &g_copy_error)) break;
    const uint8_t* src;
    uint8_t* dst;
    uint32_t bytes;
    chunk(i, src, dst, bytes);
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    bulk_s2g(dst, sbuf + (uint32_t)k * kCopyChunk, bytes);
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
    if (issued < c1) {
      // buffer k is reloaded once the store just issued has read it
      asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
      chunk(issued, src, dst, bytes);
      pipe::mbar_arrive_tx(sbar + 8u * k, bytes);
      bulk_g2s(sbuf + (uint32_t)k * kCopyChunk, src, bytes, sbar + 8u * k);
      ++issued;
    }
  }
  // No load may still be in flight into shared memory when the CTA exits
  // (only after a wait gave up), and the stores must have completed.
  for (int64_t v = i; v < issued; ++v)
    pipe::wait_bar_quiet(sbar + 8u * (uint32_t)((v - c0) % kCopyBufs), (uint32_t)(((v - c0) / kCopyBufs) & 1));
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// Exact dequantize (PR #2629 "ROCm native NVFP4", Summary: the dequantize
// kernel expands a plane exactly; Changes during review: the grid is sized
// from the weight plane). One thread-iteration expands one packed word (half
// of a 16-column block): eight outputs from the word and its block's scale
// byte, so that a warp's output store is 32 x 16 contiguous bytes (bf16/f16).
// Element value = cast(f32(fp4 * e4m3) * factor) with factor = gs[e] / 2688
// (absent gs: the product itself, exact in every output type).
template <typename OutT>
__device__ __forceinline__ void store8(OutT* dst, const uint32_t (&h)[4], float fac, bool has_gs);

__device__ __forceinline__ float h_lo(uint32_t v) { return __half2float(__ushort_as_half((unsigned short)(v & 0xFFFF))); }
__device__ __forceinline__ float h_hi(uint32_t v) { return __half2float(__ushort_as_half((unsigned short)(v >> 16))); }

template <>
__device__ __forceinline__ void store8<float>(float* dst, const uint32_t (&h)[4], float fac, bool has_gs) {
  float v[8];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[2 * i] = h_lo(h[i]);
    v[2 * i + 1] = h_hi(h[i]);
  }
  if (has_gs) {
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = __fmul_rn(v[i], fac);
  }
  uint4* d = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int q = 0; q < 2; ++q)
    __stcs(d + q, make_uint4(__float_as_uint(v[4 * q]), __float_as_uint(v[4 * q + 1]),
                             __float_as_uint(v[4 * q + 2]), __float_as_uint(v[4 * q + 3])));
}

template <>
__device__ __forceinline__ void store8<__half>(__half* dst, const uint32_t (&h)[4], float fac, bool has_gs) {
  uint32_t o[4];
  if (!has_gs) {
#pragma unroll
    for (int i = 0; i < 4; ++i) o[i] = h[i];
  } else {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const __half lo = __float2half_rn(__fmul_rn(h_lo(h[i]), fac));
      const __half hi = __float2half_rn(__fmul_rn(h_hi(h[i]), fac));
      o[i] = (uint32_t)__half_as_ushort(lo) | ((uint32_t)__half_as_ushort(hi) << 16);
    }
  }
  __stcs(reinterpret_cast<uint4*>(dst), make_uint4(o[0], o[1], o[2], o[3]));
}

template <>
__device__ __forceinline__ void store8<__nv_bfloat16>(__nv_bfloat16* dst, const uint32_t (&h)[4], float fac,
                                                      bool has_gs) {
  uint32_t o[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float a = h_lo(h[i]), b = h_hi(h[i]);
    if (has_gs) {
      a = __fmul_rn(a, fac);
      b = __fmul_rn(b, fac);
    }
    o[i] = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(a)) |
           ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(b)) << 16);
  }
  __stcs(reinterpret_cast<uint4*>(dst), make_uint4(o[0], o[1], o[2], o[3]));
}

template <typename OutT>
__global__ void __launch_bounds__(kStreamThreads)
dequantize_kernel(const uint32_t* __restrict__ w, const uint8_t* __restrict__ scales,
                  const float* __restrict__ gs, int64_t E, int64_t words_per_expert,
                  OutT* __restrict__ out) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t e = blockIdx.y; e < E; e += gridDim.y) {
    const float fac = global_factor(gs, e);
    const bool has_gs = gs != nullptr;
    const int64_t base = e * words_per_expert;  // first word of expert e
    // kU words per thread and iteration, all loads issued before any decode
    // so that their latencies overlap.
    constexpr int kU = 8;
    int64_t vi = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    for (; vi + (kU - 1) * stride < words_per_expert; vi += kU * stride) {
      uint32_t wv[kU], sb[kU];
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int64_t v = base + vi + u * stride;
        wv[u] = __ldcs(w + v);
        sb[u] = __ldcs(scales + (v >> 1));
      }
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int64_t v = base + vi + u * stride;
        uint32_t h[4];
        decode8_scaled_f16(wv[u], e4m3_to_f16x2_bcast(sb[u]), h);
        store8<OutT>(out + 8 * v, h, fac, has_gs);
      }
    }
    for (; vi < words_per_expert; vi += stride) {
      const int64_t v = base + vi;
      uint32_t h[4];
      decode8_scaled_f16(__ldcs(w + v), e4m3_to_f16x2_bcast(__ldcs(scales + (v >> 1))), h);
      store8<OutT>(out + 8 * v, h, fac, has_gs);
    }
  }
}

// ---------------------------------------------------------------- quantize
//
// Dense -> NVFP4 (the encoding half of MLX's global-scale convention, mlx PR
// #2629, Implementation Review Summary: block scales are encoded times
// 448 * 6 / global_scale). Per 16-column block, in IEEE float32:
// amax = max |x|, s = amax / 6 (times 2688 / gs with a global scale), scale
// byte = E4M3 nearest to s (ties to even, saturating at 448), d = e4m3 * gs /
// 2688, r = 1 / d, code = E2M1 nearest to x * r (ties to even, saturating at
// +-6), +0 for a zero magnitude, all codes 0 where d == 0. Both roundings are
// the hardware conversions (cvt.rn.satfinite); one reciprocal per block
// instead of a division per element keeps the kernel bound by HBM.

__device__ __forceinline__ uint32_t f32_to_e4m3_satfinite(float v) {
  unsigned short h;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(h) : "f"(0.0f), "f"(v));
  return (uint32_t)h & 0xFFu;
}

// One 16-column block's inputs as raw 16-byte words (four for f32).
template <typename T> struct Raw16 { uint4 q[sizeof(T) == 4 ? 4 : 2]; };

// Cached loads: a warp's 16-byte loads each cover every other 16 (or 48)
// bytes of its span, and the lines they bring into L1 serve the thread's
// next load (with evict-first loads: 91.9 against 90.3 us on the bf16
// gate/up plane, 172 against 167 with f32 input).
template <typename T>
__device__ __forceinline__ void load_raw16(const T* p, Raw16<T>& r) {
#pragma unroll
  for (int i = 0; i < (int)(sizeof(r.q) / sizeof(uint4)); ++i) r.q[i] = __ldg(reinterpret_cast<const uint4*>(p) + i);
}

__device__ __forceinline__ uint32_t u4get(const uint4& v, int i) { return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w; }

// The block's sixteen values as eight f32 pairs (columns 2i, 2i + 1), and
// max |x| over them. For 16-bit inputs the maximum is taken on the packed
// halves (|x| by clearing the sign bits, then a packed max: exact), one
// widening at the end.
template <typename T> __device__ __forceinline__ float widen16(const Raw16<T>& r, float (&lo)[8], float (&hi)[8]);
template <> __device__ __forceinline__ float widen16<float>(const Raw16<float>& r, float (&lo)[8], float (&hi)[8]) {
  float am = 0.0f;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    lo[i] = __uint_as_float(u4get(r.q[i >> 1], 2 * (i & 1)));
    hi[i] = __uint_as_float(u4get(r.q[i >> 1], 2 * (i & 1) + 1));
    am = fmaxf(am, fmaxf(fabsf(lo[i]), fabsf(hi[i])));
  }
  return am;
}
template <> __device__ __forceinline__ float widen16<__nv_bfloat16>(const Raw16<__nv_bfloat16>& r, float (&lo)[8],
                                                                   float (&hi)[8]) {
  uint32_t m = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint32_t u = u4get(r.q[i >> 2], i & 3);
    lo[i] = __uint_as_float(u << 16);
    hi[i] = __uint_as_float(u & 0xFFFF0000u);
    asm("max.bf16x2 %0, %0, %1;" : "+r"(m) : "r"(u & 0x7FFF7FFFu));
  }
  return fmaxf(__uint_as_float(m << 16), __uint_as_float(m & 0xFFFF0000u));
}
template <> __device__ __forceinline__ float widen16<__half>(const Raw16<__half>& r, float (&lo)[8], float (&hi)[8]) {
  uint32_t m = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint32_t u = u4get(r.q[i >> 2], i & 3);
    lo[i] = __half2float(__ushort_as_half((unsigned short)(u & 0xFFFFu)));
    hi[i] = __half2float(__ushort_as_half((unsigned short)(u >> 16)));
    asm("max.f16x2 %0, %0, %1;" : "+r"(m) : "r"(u & 0x7FFF7FFFu));
  }
  return fmaxf(__half2float(__ushort_as_half((unsigned short)(m & 0xFFFFu))),
               __half2float(__ushort_as_half((unsigned short)(m >> 16))));
}

// (a, b) * (r, r), each product rounded to nearest (one packed multiply).
__device__ __forceinline__ void mul2_rn(float& a, float& b, float r) {
  uint64_t p, q, d;
  asm("mov.b64 %0, {%1, %2};" : "=l"(p) : "f"(a), "f"(b));
  asm("mov.b64 %0, {%1, %1};" : "=l"(q) : "f"(r));
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(p), "l"(q));
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(d));
}

// Four (low, high) pairs -> one word of eight E2M1 codes, low column in the
// low nibble (cvt puts its first source in the high nibble).
__device__ __forceinline__ uint32_t cvt_e2m1x8(const float* lo, const float* hi) {
  uint32_t r;
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
      "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
      : "=r"(r)
      : "f"(lo[0]), "f"(hi[0]), "f"(lo[1]), "f"(hi[1]), "f"(lo[2]), "f"(hi[2]), "f"(lo[3]), "f"(hi[3]));
  return r;
}
// +0 for every zero magnitude (a negative value that rounds to zero).
__device__ __forceinline__ uint32_t plus_zero(uint32_t r) {
  const uint32_t nz = (r | (r >> 1) | (r >> 2)) & 0x11111111u;
  return (r & 0x77777777u) | (r & (nz << 3));
}

// Magnitude code of the E2M1 value nearest to the exact quotient a / d, for
// a >= 0 and d in [1, 2) (both scaled by the same power of two, which leaves
// the quotient as it is): a is compared with each midpoint m of the grid
// times d. fmaf forms a - m * d with one rounding, and with d in [1, 2) and
// a near m * d no result is small enough to underflow, so its sign is the
// exact comparison; a tie (+0) goes to the even code (up at 0.75, 1.75 and
// 3.5, down at the others). A quotient past 5 saturates at code 7 (6.0); a
// NaN compares false everywhere and gives 0.
__device__ __forceinline__ uint32_t e2m1_code_exact(float a, float d) {
  uint32_t c = 0;
  c += fmaf(-0.25f, d, a) > 0.0f;
  c += fmaf(-0.75f, d, a) >= 0.0f;
  c += fmaf(-1.25f, d, a) > 0.0f;
  c += fmaf(-1.75f, d, a) >= 0.0f;
  c += fmaf(-2.5f, d, a) > 0.0f;
  c += fmaf(-3.5f, d, a) >= 0.0f;
  c += fmaf(-5.0f, d, a) > 0.0f;
  return c;
}

// Element e (0..15, a run-time index) of a block's raw 16-byte words, as
// float.
__device__ __forceinline__ uint32_t u4sel(const uint4& v, int i) {
  const uint32_t a = (i & 1) ? v.y : v.x, b = (i & 1) ? v.w : v.z;
  return (i & 2) ? b : a;
}
template <typename T> __device__ __forceinline__ float raw_elem(const Raw16<T>& r, int e);
template <> __device__ __forceinline__ float raw_elem<float>(const Raw16<float>& r, int e) {
  const uint4 q = (e & 8) ? ((e & 4) ? r.q[3] : r.q[2]) : ((e & 4) ? r.q[1] : r.q[0]);
  return __uint_as_float(u4sel(q, e & 3));
}
template <> __device__ __forceinline__ float raw_elem<__nv_bfloat16>(const Raw16<__nv_bfloat16>& r, int e) {
  const uint32_t u = u4sel((e & 8) ? r.q[1] : r.q[0], (e & 7) >> 1);
  return __uint_as_float((e & 1) ? (u & 0xFFFF0000u) : (u << 16));
}
template <> __device__ __forceinline__ float raw_elem<__half>(const Raw16<__half>& r, int e) {
  const uint32_t u = u4sel((e & 8) ? r.q[1] : r.q[0], (e & 7) >> 1);
  return __half2float(__ushort_as_half((unsigned short)((e & 1) ? (u >> 16) : (u & 0xFFFFu))));
}

// Power-of-two scaling of a block's comparisons: |x| and d are multiplied by
// 2^-E, d = dn 2^E with dn in [1, 2), which leaves every quotient as it is.
// It is exact, except that an |x| far below d may lose bits (it stays below
// every midpoint) and one far above may become infinite (it stays above). A
// d below 2^-126 (a float32 subnormal) is first scaled by 2^126, and |x| with
// it, one power of two after the other.
struct Scaled {
  float pre, p, dn;
  __device__ __forceinline__ explicit Scaled(float d) {
    pre = d < 0x1p-126f ? 0x1p126f : 1.0f;
    const uint32_t db = __float_as_uint(d * pre);
    dn = __uint_as_float((db & 0x007FFFFFu) | 0x3F800000u);
    p = __uint_as_float((254u - (db >> 23)) << 23);  // 2^-E of d * pre, in [2^-125, 2^126]
  }
  __device__ __forceinline__ float operator()(float x) const { return (fabsf(x) * pre) * p; }
};

// The midpoint of E2M1 codes c and c + 1 (0.25, 0.75, 1.25, 1.75, 2.5, 3.5,
// 5 for c = 0..6): the float32 bits 0x3E800000 + (v << 21) with v = 0, 6, 9,
// 11, 13, 15, 17, five bits each in one 64-bit constant.
__device__ __forceinline__ float e2m1_midpoint(uint32_t c) {
  constexpr uint64_t kV = 0ull | (6ull << 5) | (9ull << 10) | (11ull << 15) | (13ull << 20) | (15ull << 25) |
                          (17ull << 30);
  return __uint_as_float(0x3E800000u + ((((uint32_t)(kV >> (5 * c))) & 31u) << 21));
}

// The values whose two conversions disagree (set nibbles of dm, elements e0
// .. e0 + 7 of the block, codes of the upper products in hw). The products
// lie within a factor 1 + 2^-20 of each other and the midpoints at least a
// factor 1.4 apart, so exactly one midpoint m separates the two codes (c from
// the lower product, c + 1 from the upper one): the sign of |x| - m d picks
// one of them, and a tie the even one. fmaf forms |x| - m d with one
// rounding; for d >= 2^-100 (callers send smaller d to exact_block) no
// nonzero result of it underflows to zero, so its sign is the exact
// comparison. The result still needs plus_zero.
template <typename T>
__device__ __forceinline__ uint32_t fix_codes(uint32_t hw, uint32_t dm, const Raw16<T>& r, int e0, float d) {
  const uint32_t lw = hw ^ dm;
  while (dm) {
    const int sh = (__ffs(dm) - 1) & ~3;
    dm &= ~(0xFu << sh);
    const uint32_t c = (lw >> sh) & 7u;
    const float t = fmaf(-e2m1_midpoint(c), d, fabsf(raw_elem<T>(r, e0 + (sh >> 2))));
    const bool up = t > 0.0f || (t == 0.0f && (c & 1u));
    hw = (hw & ~(0xFu << sh)) | ((((up ? hw : lw) >> sh) & 0xFu) << sh);
  }
  return hw;
}

// Every code of a block by the full comparisons (a d whose reciprocal
// overflows float32). A zero magnitude gets +0.
template <typename T>
__device__ __forceinline__ uint2 exact_block(const Raw16<T>& r, float d) {
  const Scaled sc(d);
  uint32_t wd[2] = {0u, 0u};
  for (int e = 0; e < 16; ++e) {
    const float x = raw_elem<T>(r, e);
    const uint32_t c = e2m1_code_exact(sc(x), sc.dn);
    const uint32_t nib = c | (c != 0u && x < 0.0f ? 8u : 0u);
    wd[e >> 3] |= nib << (4 * (e & 7));
  }
  return make_uint2(wd[0], wd[1]);
}

// One 16-column block (two output words and a scale byte) per thread and
// step, four blocks in flight (128 or 256 bytes of loads a thread). The code
// of each value is the E2M1 value nearest to the exact |x| / d.
template <typename T>
__global__ void __launch_bounds__(kStreamThreads)
quantize_kernel(const T* __restrict__ x, const float* __restrict__ gs, int64_t E, int64_t blocks_per_expert,
                uint32_t* __restrict__ w, uint8_t* __restrict__ scales) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  const int64_t first = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  for (int64_t e = blockIdx.y; e < E; e += gridDim.y) {
    const bool has_gs = gs != nullptr;
    const float fac = global_factor(gs, e);
    const float inv = has_gs ? __fdiv_rn(kGlobalScaleDivisor, __ldg(gs + e)) : 1.0f;
    const int64_t base = e * blocks_per_expert;
    constexpr int kU = 4;
    for (int64_t b0 = first; b0 < blocks_per_expert; b0 += kU * stride) {
      Raw16<T> raw[kU];
#pragma unroll
      for (int k = 0; k < kU; ++k) {
        const int64_t b = b0 + k * stride;
        if (b < blocks_per_expert) load_raw16<T>(x + 16 * (base + b), raw[k]);
      }
#pragma unroll
      for (int k = 0; k < kU; ++k) {
        const int64_t b = b0 + k * stride;
        if (b >= blocks_per_expert) break;
        float lo[8], hi[8];
        const float am = widen16<T>(raw[k], lo, hi);
        float sc = __fdiv_rn(am, 6.0f);
        if (has_gs) sc = __fmul_rn(sc, inv);
        const uint32_t sbyte = f32_to_e4m3_satfinite(sc);
        const float d = __fmul_rn(e4m3_to_f32(sbyte), fac);
        uint2 out = make_uint2(0u, 0u);
        if (d > 0.0f) {
          // Each value is converted twice, from x * r (1 - 2^-21) and
          // x * r (1 + 2^-21): the product x * r is within two roundings
          // (2^-23 relative) of the quotient x / d, so the quotient lies
          // between the two products, and where both convert to the same
          // code (the nearest-value code is monotone) that code is the one
          // of the quotient. Codes that differ (a midpoint lies between the
          // products) take the exact comparisons.
          const float r = __frcp_rn(d);
          const float rl = __fmul_rn(r, 1.0f - 0x1p-21f), rh = __fmul_rn(r, 1.0f + 0x1p-21f);
          float ll[8], lh[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            ll[i] = lo[i];
            lh[i] = hi[i];
            mul2_rn(lo[i], hi[i], rh);
            mul2_rn(ll[i], lh[i], rl);
          }
          uint32_t hx = cvt_e2m1x8(lo, hi), hy = cvt_e2m1x8(lo + 4, hi + 4);
          const uint32_t dx = hx ^ cvt_e2m1x8(ll, lh), dy = hy ^ cvt_e2m1x8(ll + 4, lh + 4);
          if (dx) hx = fix_codes<T>(hx, dx, raw[k], 0, d);
          if (dy) hy = fix_codes<T>(hy, dy, raw[k], 8, d);
          out = make_uint2(plus_zero(hx), plus_zero(hy));
          // d below 2^-100: the comparisons need scaling (and below 2^-127
          // the reciprocal overflows)
          if (d < 0x1p-100f) out = exact_block<T>(raw[k], d);
        }
        __stcs(reinterpret_cast<uint2*>(w) + base + b, out);
        scales[base + b] = (uint8_t)sbyte;
      }
    }
  }
}

// ---------------------------------------------------------------- folded-scale transcode
//
// The alternative that issue #693 (Technical notes) rejects, built to measure
// what it loses: weight_scale * weight_scale_2 folded into each E4M3 byte, no
// sidecar. Weight bytes are copied as they are (the word plane is the byte
// stream); each scale byte becomes the E4M3 nearest to f32(e4m3(b) * ws2),
// ties to even, saturating at 448, small products flushed to 0 or a
// subnormal.

__device__ __forceinline__ uint32_t fold_byte(uint32_t b, float ws2) {
  return f32_to_e4m3_satfinite(__fmul_rn(e4m3_to_f32(b & 0xFFu), ws2));
}

__device__ __forceinline__ uint32_t fold_word(uint32_t v, float ws2) {
  return fold_byte(v, ws2) | (fold_byte(v >> 8, ws2) << 8) | (fold_byte(v >> 16, ws2) << 16) |
         (fold_byte(v >> 24, ws2) << 24);
}

__global__ void __launch_bounds__(kStreamThreads)
transcode_folded_kernel(const uint8_t* __restrict__ mo_w, int64_t w_bytes, const uint8_t* __restrict__ mo_ws,
                        int64_t s_bytes, const float* __restrict__ ws2p, uint8_t* __restrict__ w_out,
                        uint8_t* __restrict__ s_out) {
  const float ws2 = __ldg(ws2p);
  const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  const int64_t wv = w_bytes >> 4, sv = s_bytes >> 4;
  const uint4* wi = reinterpret_cast<const uint4*>(mo_w);
  uint4* wo = reinterpret_cast<uint4*>(w_out);
  constexpr int kU = 4;  // loads in flight per thread
  int64_t i = tid;
  for (; i + (kU - 1) * stride < wv; i += kU * stride) {
    uint4 v[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) v[u] = __ldcs(wi + i + u * stride);
#pragma unroll
    for (int u = 0; u < kU; ++u) __stcs(wo + i + u * stride, v[u]);
  }
  for (; i < wv; i += stride) __stcs(wo + i, __ldcs(wi + i));
  const uint4* si = reinterpret_cast<const uint4*>(mo_ws);
  uint4* so = reinterpret_cast<uint4*>(s_out);
  for (int64_t j = tid; j < sv; j += stride) {
    const uint4 v = __ldcs(si + j);
    __stcs(so + j, make_uint4(fold_word(v.x, ws2), fold_word(v.y, ws2), fold_word(v.z, ws2), fold_word(v.w, ws2)));
  }
  for (int64_t j = (wv << 4) + tid; j < w_bytes; j += stride) w_out[j] = mo_w[j];
  for (int64_t j = (sv << 4) + tid; j < s_bytes; j += stride) s_out[j] = (uint8_t)fold_byte(mo_ws[j], ws2);
}

}  // namespace

cudaError_t launch_transcode(const uint8_t* mo_w, int64_t w_bytes, const uint8_t* mo_ws, int64_t s_bytes,
                             const float* ws2, uint32_t* w_out, uint8_t* s_out, float* gs_out,
                             cudaStream_t st) {
  int dev = 0, sms = 152;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const size_t smem = (size_t)kCopyBufs * kCopyChunk;
  cudaError_t e = cudaFuncSetAttribute(transcode_bulk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  transcode_bulk_kernel<<<sms, 32, smem, st>>>(mo_w, w_bytes, mo_ws, s_bytes, ws2, reinterpret_cast<uint8_t*>(w_out),
                                              s_out, gs_out);
  return cudaGetLastError();
}

cudaError_t launch_quantize(const void* x, int x_dtype, const float* gs, int64_t E, int64_t N, int64_t K,
                            uint32_t* w, uint8_t* scales, cudaStream_t st) {
  const int64_t bpe = N * (K / 16);  // 16-column blocks per expert
  auto grid_of = [&](auto kern) {
    int gx = stream_grid(kern, (bpe * E + 1) / 2);
    const int64_t per_expert = (bpe + kStreamThreads - 1) / kStreamThreads;
    if (gx > per_expert) gx = (int)(per_expert < 1 ? 1 : per_expert);
    const int gy = (int)(E < 65535 ? E : 65535);
    return dim3(gx, gy);
  };
  switch (x_dtype) {
    case kF32:
      quantize_kernel<float><<<grid_of(quantize_kernel<float>), kStreamThreads, 0, st>>>(
          static_cast<const float*>(x), gs, E, bpe, w, scales);
      break;
    case kF16:
      quantize_kernel<__half><<<grid_of(quantize_kernel<__half>), kStreamThreads, 0, st>>>(
          static_cast<const __half*>(x), gs, E, bpe, w, scales);
      break;
    default:
      quantize_kernel<__nv_bfloat16><<<grid_of(quantize_kernel<__nv_bfloat16>), kStreamThreads, 0, st>>>(
          static_cast<const __nv_bfloat16*>(x), gs, E, bpe, w, scales);
      break;
  }
  return cudaGetLastError();
}

cudaError_t launch_transcode_folded(const uint8_t* mo_w, int64_t w_bytes, const uint8_t* mo_ws, int64_t s_bytes,
                                    const float* ws2, uint32_t* w_out, uint8_t* s_out, cudaStream_t st) {
  const int64_t units = (w_bytes >> 4) / 4 + (s_bytes >> 4) + 16;
  transcode_folded_kernel<<<stream_grid(transcode_folded_kernel, units), kStreamThreads, 0, st>>>(
      mo_w, w_bytes, mo_ws, s_bytes, ws2, reinterpret_cast<uint8_t*>(w_out), s_out);
  return cudaGetLastError();
}

int read_copy_error() {
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_copy_error, sizeof(int)) != cudaSuccess) return -1;
  const int zero = 0;
  cudaMemcpyToSymbol(g_copy_error, &zero, sizeof(int));
  return v;
}

cudaError_t launch_dequantize(const uint32_t* w, const uint8_t* scales, const float* gs, int64_t E,
                              int64_t N, int64_t K, int out_dtype, void* out, cudaStream_t st) {
  const int64_t gpe = N * (K / 8);  // words per expert
  auto grid_of = [&](auto kern) {
    int gx = stream_grid(kern, (gpe * E + 7) / 8);
    const int64_t per_expert = (gpe + kStreamThreads - 1) / kStreamThreads;
    if (gx > per_expert) gx = (int)(per_expert < 1 ? 1 : per_expert);
    const int gy = (int)(E < 65535 ? E : 65535);
    return dim3(gx, gy);
  };
  switch (out_dtype) {
    case kF32:
      dequantize_kernel<float><<<grid_of(dequantize_kernel<float>), kStreamThreads, 0, st>>>(w, scales, gs, E, gpe,
                                                                                            (float*)out);
      break;
    case kF16:
      dequantize_kernel<__half><<<grid_of(dequantize_kernel<__half>), kStreamThreads, 0, st>>>(w, scales, gs, E, gpe,
                                                                                              (__half*)out);
      break;
    default:
      dequantize_kernel<__nv_bfloat16><<<grid_of(dequantize_kernel<__nv_bfloat16>), kStreamThreads, 0, st>>>(
          w, scales, gs, E, gpe, (__nv_bfloat16*)out);
      break;
  }
  return cudaGetLastError();
}

}  // namespace nvfp4
